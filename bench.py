#!/usr/bin/env python3
"""Benchmark of the TokenGate gated-prefill hot path on one B300.

One step = one pass of the whole path over one batch:
  gate score (K1) -> top-K select (K2) -> gather kept rows (K3) -> gated attention (K4)
over synthetic inputs shaped like the Qwen3-1.7B long-context prefill of the TokenGate pages
(default: B=1, N = 32768 document + 256 instruction tokens, d=2048, d_g=512, 16/8 heads of
128, budget K=4096). Tokens = all tokens entering the gate layer.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--k K]
  python bench.py --impl reference ...   # the CPU oracle, timed on a bounded sample

Prints one JSON line (rank 0). With N > 1 (torchrun) every rank runs an independent replica
on its own seeded batch (the path shards over independent sequences; there is no collective
on the data path) and the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "gated-prefill tokens/s (score+topK+gather+gated attn), N=32K; % of roofline"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 256 << 20
L2_NOTE = ("flushed between timed steps, outside the per-step events: a 256 MB write, then a 256 MB read of a "
           "second buffer, so the step's inputs start in HBM and L2 holds no dirty lines for the first kernel")


class L2Flush:
    """Evicts the step's inputs from the 126 MB L2 between timed steps: a write of one buffer larger
    than L2, then a read of a second one, which also writes back the first buffer's dirty lines
    before the next step starts (otherwise the first kernel of the step pays for that write-back)."""

    def __init__(self, torch):
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
        self.sink = torch.empty(1, dtype=torch.float32, device="cuda")

    def __call__(self):
        self.w.zero_()
        self.sink.copy_(self.r.sum().reshape(1))
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "ncu_traffic.txt")


# ---------------------------------------------------------------------------
# distributed plumbing (host logic; covered by gloo tests on CPU)
# ---------------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def replica_seed(base_seed: int, rank: int) -> int:
    """Each rank processes its own independent batch (weak scaling)."""
    return base_seed + 1000 * rank


def reduce_max(value: float, world: int) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(tokens_per_rank: int, world: int, max_seconds: float) -> float:
    """Whole-job throughput: the tokens all ranks processed over the slowest rank's time."""
    return tokens_per_rank * world / max_seconds


# ---------------------------------------------------------------------------
# algorithmic work per stage (the roofline numerators)
# ---------------------------------------------------------------------------

def stage_work(wl, K: int, kept_lens):
    T, d, d_g = wl.T_total, wl.d, wl.d_g
    M = int(sum(kept_lens))
    B = wl.B
    attn_pairs = sum(m * (m + 1) // 2 for m in kept_lens)
    return {
        "gate_score": {"bound": "tensor", "flops": 2.0 * T * d * d_g,
                       "bytes": T * d * 2 + d_g * d * 2 + T * (1 + 4 + 4)},
        "topk_select": {"bound": "hbm", "bytes": T * 4 + T * 1 + M * 4 + 2 * (B + 1) * 4},
        "gather_kept": {"bound": "hbm", "bytes": 2 * M * d * 2 + M * 4 + 2 * M * 4 + 2 * M * 4},
        "gated_attention": {"bound": "tensor", "flops": 4.0 * wl.d_h * wl.H_q * attn_pairs,
                            "bytes": M * (wl.H_q + 2 * wl.H_kv) * wl.d_h * 2 + M * 4 + M * wl.H_q * wl.d_h * 2},
    }


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": float(j["hbm_gbs"]), "bf16_tflops": float(j["bf16_tflops"]),
                "bf16_tflops_sustained": float(j.get("bf16_tflops_sustained", j["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


def strip_comments(src: str) -> str:
    """C++ source without its comments and blank lines, so a comment-only edit keeps the hash."""
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(line.rstrip() for line in src.splitlines() if line.strip())


def kernel_source_hash(name: str) -> str:
    """Hash of the code (comments stripped) of a kernel's source file and the common header."""
    files = {"gate_score": "tg_score.cu", "topk_select": "tg_select.cu", "gather_kept": "tg_gather.cu",
             "gated_attention": "tg_attention.cu"}
    h = hashlib.sha256()
    for f in (files[name], "tg_common.cuh"):
        with open(os.path.join(ROOT, "learned_token_pruning_07_b300", "csrc", f), encoding="utf-8") as fh:
            h.update(strip_comments(fh.read()).encode())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, workload: str, K: int):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on this exact
    kernel source and workload; otherwise None."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    with open(PROFILE_TRAFFIC) as f:
        for line in f:
            parts = line.split()
            if len(parts) != 5 or line.startswith("#") or parts[0] != kernel:
                continue
            if parts[1] == workload and int(parts[2]) == K and parts[3] == kernel_source_hash(kernel):
                return float(parts[4])
    return None


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# the GPU path
# ---------------------------------------------------------------------------

class GatedPrefill:
    """Device buffers for one batch and the step that runs the four kernels on them."""

    def __init__(self, wl, K, torch):
        from learned_token_pruning_07_b300 import binding as tg
        from learned_token_pruning_07_b300 import inputs as I
        self.tg, self.I, self.torch = tg, I, torch
        self.wl, self.K = wl, K
        gi = I.make_gate_inputs(wl)
        self.kept_lens = [min(K, a) + b for a, b in zip(wl.doc_lens, wl.instr_lens)]
        self.M = int(sum(self.kept_lens))
        self.max_seqlen = max(self.kept_lens)
        at = I.make_attention_inputs(wl, self.M)
        self.tau, self.beta = at["tau"], at["beta"]
        T, B = wl.T_total, wl.B

        def pinned(a):
            a = np.ascontiguousarray(a)
            t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
            return t.pin_memory()

        # host copies (pinned) of the step's activations, for the end-to-end leg
        self.host = {k: pinned(v) for k, v in (("h", gi["h"]), ("mask", gi["instr_mask"]),
                                               ("cu", gi["cu_seqlens"]), ("pos", gi["pos"]),
                                               ("Q", at["Q"]), ("K", at["K"]), ("V", at["V"]))}
        dev = lambda t: t.to("cuda", non_blocking=False)
        self.d = {k: dev(v) for k, v in self.host.items()}
        self.W1 = dev(pinned(gi["W1"]))
        self.w2 = dev(pinned(gi["w2"]))
        e = lambda *shape, dt=torch.float32: torch.empty(*shape, dtype=dt, device="cuda")
        self.s, self.g = e(T), e(T)
        # the tie-heavy workload selects from its synthetic 256-level score buffer; the others rank
        # the scores the step itself computes
        self.s_sel = self.s if not wl.score_levels else torch.from_numpy(I.make_scores(wl)).cuda()
        self.kept, self.cu_kept = e(T, dt=torch.int32), e(B + 1, dt=torch.int32)
        self.h_kept = e(T, wl.d, dt=torch.int16)
        self.pos_kept, self.g_kept = e(T, dt=torch.int32), e(T)
        self.O = e(self.M, wl.H_q, wl.d_h, dt=torch.int16)
        # attention workspace: used when one CTA per query tile would leave SMs idle (short kept
        # sequences); empty otherwise. Zero-filled once; each call leaves it zeroed.
        self.ws = tg.attention_workspace(B, self.max_seqlen, wl.H_q, wl.H_kv, wl.d_h)
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.O_host = torch.empty(self.O.shape, dtype=torch.int16).pin_memory()
        self.cu_kept_host = torch.empty(B + 1, dtype=torch.int32).pin_memory()

    def step(self, ev=(None,) * 5):
        """K1..K4 on device-resident inputs; ev = 5 events (or None) recorded around the kernels.
        An event between two kernels also separates them (no launch overlap across it)."""
        tg, d = self.tg, self.d
        rec = lambda e: e.record() if e is not None else None
        rec(ev[0])
        tg.gate_score(d["h"], self.W1, self.w2, self.s, self.g, instr_mask=d["mask"], status=self.status)
        rec(ev[1])
        tg.topk_select(self.s_sel, d["cu"], self.K, self.kept, self.cu_kept, instr_mask=d["mask"],
                       status=self.status)
        rec(ev[2])
        tg.gather_kept(d["h"], d["cu"], self.kept, self.cu_kept, self.h_kept, pos=d["pos"], g=self.g,
                       pos_kept=self.pos_kept, g_kept=self.g_kept, status=self.status)
        rec(ev[3])
        tg.gated_attention(d["Q"], d["K"], d["V"], self.cu_kept, self.tau, self.beta, self.O,
                           max_seqlen=self.max_seqlen, g=self.g_kept, status=self.status, workspace=self.ws)
        rec(ev[4])

    def step_e2e(self):
        """The public fused call with host buffers: H2D of the step's activations, the path,
        D2H of the attention output and the kept counts."""
        tg, d, h = self.tg, self.d, self.host
        for k in ("h", "mask", "cu", "pos", "Q", "K", "V"):
            d[k].copy_(h[k], non_blocking=True)
        tg.gate_prune_layer(d["h"], d["cu"], self.W1, self.w2, self.K, self.s, self.g, self.kept, self.cu_kept,
                            self.h_kept, pos_kept=self.pos_kept, g_kept=self.g_kept, pos=d["pos"],
                            instr_mask=d["mask"], status=self.status)
        tg.gated_attention(d["Q"], d["K"], d["V"], self.cu_kept, self.tau, self.beta, self.O,
                           max_seqlen=self.max_seqlen, g=self.g_kept, status=self.status, workspace=self.ws)
        self.O_host.copy_(self.O, non_blocking=True)
        self.cu_kept_host.copy_(self.cu_kept, non_blocking=True)

    def h2d_bytes(self):
        return sum(self.host[k].numel() * self.host[k].element_size() for k in ("h", "mask", "cu", "pos", "Q", "K", "V"))

    def d2h_bytes(self):
        return self.O_host.numel() * 2 + self.cu_kept_host.numel() * 4


class GraphStep:
    """The four-kernel step captured once in CUDA graphs, so host launch overhead never shows
    up on the device timeline. Two graphs: `whole` records events only around the step, so
    each kernel's launch may overlap the previous kernel's tail (programmatic dependent
    launch) -- this one gives the step time; `staged` records an event between every two
    kernels and gives the per-kernel breakdown. A third, `paired`, has no event between the
    selection and the gather, so the pair is timed as the fused call runs it (the gather's
    launch overlapping the selection's tail)."""

    def __init__(self, path, torch):
        self.torch = torch
        self.ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(5)]
        self.ew = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
        self.ep = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(4)]
        path.step()                      # first launch sets kernel attributes outside capture
        torch.cuda.synchronize()
        self.staged = self._capture(path, self.ev)
        self.whole = self._capture(path, [self.ew[0], None, None, None, self.ew[1]])
        self.paired = self._capture(path, [self.ep[0], self.ep[1], None, self.ep[2], self.ep[3]])
        self.graph = self.whole

    def _capture(self, path, ev):
        torch = self.torch
        graph = torch.cuda.CUDAGraph()
        stream = torch.cuda.Stream()
        stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            graph.capture_begin(capture_error_mode="relaxed")
            path.step(ev)
            graph.capture_end()
        torch.cuda.current_stream().wait_stream(stream)
        torch.cuda.synchronize()
        return graph

    def replay(self, staged=False):
        (self.staged if staged else self.whole).replay()

    def pair_time(self):
        return self.ep[1].elapsed_time(self.ep[2])

    def step_time(self):
        return self.ew[0].elapsed_time(self.ew[1])

    def times(self):
        e = self.ev
        return [e[k].elapsed_time(e[k + 1]) for k in range(4)]


def warm(gstep, warmup, torch, flush):
    for _ in range(warmup):
        gstep.replay()
        flush()
        gstep.replay(staged=True)
        flush()
    torch.cuda.synchronize()


def time_whole_steps(gstep, steps, torch, flush):
    """One replay of the whole-step graph per step; L2 is flushed between steps (outside the
    events) and each step's time is read before the next."""
    per_step = []
    for _ in range(steps):
        flush()
        gstep.replay()
        torch.cuda.synchronize()
        per_step.append(gstep.step_time())
    return np.array(per_step)


def time_stages(gstep, steps, torch, flush):
    """The per-kernel breakdown: replays of the staged graph, L2 flushed between steps."""
    per_stage = []
    for _ in range(steps):
        flush()
        gstep.replay(staged=True)
        torch.cuda.synchronize()
        per_stage.append(gstep.times())
    return np.array(per_stage)


def time_pairs(gstep, steps, torch, flush):
    """Selection + gather with no event between them (the `paired` graph), L2 flushed between steps."""
    out = []
    for _ in range(steps):
        flush()
        gstep.paired.replay()
        torch.cuda.synchronize()
        out.append(gstep.pair_time())
    return np.array(out)


def time_device_steps(gstep, steps, torch, flush):
    return time_whole_steps(gstep, steps, torch, flush), time_stages(gstep, steps, torch, flush)


def time_e2e(path, steps, warmup, torch):
    for _ in range(warmup):
        path.step_e2e()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        path.step_e2e()
        b.record()
        b.synchronize()  # the host holds the step's result
        times.append(a.elapsed_time(b))
    return np.array(times)


# ---------------------------------------------------------------------------
# the CPU oracle, timed on a bounded sample
# ---------------------------------------------------------------------------

def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else (os.cpu_count() or 1)
    except Exception:
        return os.cpu_count() or 1


def _oracle_inputs(wl, K, cache):
    """The step's seeded inputs, widened once for the oracle (not timed)."""
    from learned_token_pruning_07_b300 import inputs as I
    if "gi" not in cache:
        gi = I.make_gate_inputs(wl)
        cache["gi"] = gi
        cache["h64"] = I.bf16_bits_to_f64(gi["h"])
        cache["W1"] = I.bf16_bits_to_f64(gi["W1"])
        cache["w2"] = I.bf16_bits_to_f64(gi["w2"])
        kept_lens = [min(K, a) + b for a, b in zip(wl.doc_lens, wl.instr_lens)]
        at = I.make_attention_inputs(wl, sum(kept_lens))
        cache["at"] = {k: (I.bf16_bits_to_f64(v) if k in ("Q", "K", "V") else v) for k, v in at.items()}
        # a workload whose selection scores are quantised (the tie-heavy ragged batch) selects
        # from its synthetic quantised buffer, as the GPU step does
        cache["s_sel"] = I.make_scores(wl) if wl.score_levels else None
    return cache


def oracle_step(wl, K, cache):
    """One whole, unsampled step of the oracle on the step's inputs: score every row, select,
    gather, then gated attention over every kept row. Returns the seconds of each stage."""
    from oracle import tokengate_oracle as O
    c = _oracle_inputs(wl, K, cache)
    gi, at = c["gi"], c["at"]
    t0 = time.perf_counter()
    s, g = O.gate_score(c["h64"], c["W1"], c["w2"], gi["instr_mask"])
    t1 = time.perf_counter()
    s_sel = c["s_sel"] if c["s_sel"] is not None else s.astype(np.float32)
    kept, cu_kept = O.topk_select(s_sel, gi["instr_mask"], gi["cu_seqlens"], K)
    t2 = time.perf_counter()
    _, _, g_kept = O.gather_kept(gi["h"], gi["pos"], g, kept, gi["cu_seqlens"])
    t3 = time.perf_counter()
    O.gated_attention(at["Q"], at["K"], at["V"], g_kept, cu_kept, at["tau"].astype(np.float64),
                      at["beta"].astype(np.float64))
    t4 = time.perf_counter()
    return {"score": t1 - t0, "select": t2 - t1, "gather": t3 - t2, "attention": t4 - t3, "step": t4 - t0}


_ONE_THREAD_ENV = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS",
                   "NUMEXPR_NUM_THREADS")


def oracle_stage_threads(wl, K, cache):
    """Score, select and gather of the oracle on every BLAS thread (this process) and on one
    thread (a child process started with the BLAS thread counts set to 1)."""
    all_cores = {k: v * 1000.0 for k, v in oracle_step_front(wl, K, cache).items()}
    env = dict(os.environ)
    env.update({k: "1" for k in _ONE_THREAD_ENV})
    code = ("import json, sys; sys.path.insert(0, %r); import bench; "
            "from learned_token_pruning_07_b300 import inputs as I; "
            "t = bench.oracle_step_front(I.WORKLOADS[%r], %d, {}); print(json.dumps(t))") % (ROOT, wl.name, K)
    single = None
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
        if r.returncode == 0:
            single = {k: v * 1000.0 for k, v in json.loads(r.stdout.strip().splitlines()[-1]).items()}
    except (OSError, subprocess.TimeoutExpired, ValueError, IndexError):
        single = None
    return {"all_cores": all_cores, "single_thread": single, "unit": "ms",
            "threads_all_cores": blas_threads()}


def oracle_step_front(wl, K, cache):
    """The oracle's score, select and gather of one step (attention left out), in seconds."""
    from oracle import tokengate_oracle as O
    c = _oracle_inputs(wl, K, cache)
    gi = c["gi"]
    t0 = time.perf_counter()
    s, g = O.gate_score(c["h64"], c["W1"], c["w2"], gi["instr_mask"])
    t1 = time.perf_counter()
    s_sel = c["s_sel"] if c["s_sel"] is not None else s.astype(np.float32)
    kept, _ = O.topk_select(s_sel, gi["instr_mask"], gi["cu_seqlens"], K)
    t2 = time.perf_counter()
    O.gather_kept(gi["h"], gi["pos"], g, kept, gi["cu_seqlens"])
    t3 = time.perf_counter()
    return {"score": t1 - t0, "select": t2 - t1, "gather": t3 - t2}


def oracle_sample_text(n_steps, spent):
    return (f"{n_steps} whole unsampled oracle step(s) of this workload (numpy fp64: every row scored, full "
            f"select and gather, attention over every kept row), {spent:.1f} s of CPU time; value = tokens / "
            f"median step time")


def cpu_baseline(wl, K, min_s=10.0, max_steps=3):
    """The oracle as it stands, timed on whole steps of the same workload (at least one, until
    min_s seconds are spent, at most max_steps), plus the single-thread and all-core times of
    its score, select and gather stages. The same measurement as the reference arm's steps."""
    cache = {}
    steps, spent = [], 0.0
    while (spent < min_s and len(steps) < max_steps) or not steps:
        t = oracle_step(wl, K, cache)
        steps.append(t)
        spent += t["step"]
    med = statistics.median([t["step"] for t in steps])
    stage_ms = {k: 1000.0 * statistics.median([t[k] for t in steps]) for k in steps[0]}
    return {"value": wl.T_total / med, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
            "ms_per_step": 1000.0 * med, "stage_ms": stage_ms,
            "front_stages_by_threads": oracle_stage_threads(wl, K, cache),
            "sample": oracle_sample_text(len(steps), spent)}


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------

def graph_timed(fn, reps, torch, flush, unit_scale=1000.0):
    """Median device time of fn's kernels: fn is captured once in a CUDA graph, then each rep
    flushes L2 and replays the graph between two events on the launching stream, so host
    launch overhead never lands inside the events. unit_scale 1000 gives microseconds."""
    fn()  # first call outside capture (sets kernel attributes)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        graph.capture_begin(capture_error_mode="relaxed")
        fn()
        graph.capture_end()
    torch.cuda.current_stream().wait_stream(stream)
    graph.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        graph.replay()
        b.record()
        b.synchronize()
        ts.append(a.elapsed_time(b) * unit_scale)
    del graph
    return float(np.median(ts))


def long_context(torch, flush, steps):
    """The 128K long-context workload: one pruned step (K = 8192) against full causal GQA
    attention over all 131,584 tokens, the attention the layers at or below the gate run."""
    from learned_token_pruning_07_b300 import inputs as I
    wl = I.WORKLOADS["long_128k"]
    path = GatedPrefill(wl, wl.K, torch)
    g = GraphStep(path, torch)
    warm(g, 3, torch, flush)
    ps, pst = time_device_steps(g, max(3, min(steps, 10)), torch, flush)
    wk = stage_work(wl, wl.K, path.kept_lens)
    del g, path
    torch.cuda.empty_cache()
    # full causal attention: seeded synthetic Q/K/V made on the device (timing only)
    M = wl.T_total
    gen = torch.Generator(device="cuda").manual_seed(wl.seed)
    Q = torch.randn((M, wl.H_q, wl.d_h), generator=gen, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    Kt = torch.randn((M, wl.H_kv, wl.d_h), generator=gen, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    V = torch.randn((M, wl.H_kv, wl.d_h), generator=gen, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    O = torch.empty_like(Q)
    cu = torch.tensor([0, M], dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tau, beta = np.ones(wl.H_q, np.float32), np.zeros(wl.H_q, np.float32)
    from learned_token_pruning_07_b300 import binding as tg
    call = lambda: tg.gated_attention(Q, Kt, V, cu, tau, beta, O, max_seqlen=M, g=None, status=st)
    call()
    torch.cuda.synchronize()
    times = []
    for _ in range(3):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        call()
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b))
    assert tg.read_device_status(st) == 0, "device reported an error"
    full_ms = float(np.median(times))
    full_flops = 4.0 * wl.d_h * wl.H_q * M * (M + 1) / 2
    del Q, Kt, V, O
    torch.cuda.empty_cache()
    pruned_attn_ms = float(pst[:, 3].mean())
    return {"workload": workload_label(wl, wl.K) + "; full causal attention over all tokens",
            "pruned_step_ms": float(ps.mean()), "pruned_tokens_per_s": wl.T_total / (float(ps.mean()) / 1000.0),
            "pruned_stage_us": [float(x) * 1000.0 for x in pst.mean(axis=0)], "stage_names": STAGE_NAMES,
            "pruned_attention_tflops": wk["gated_attention"]["flops"] / (pruned_attn_ms * 1e-3) / 1e12,
            "full_attention_ms": full_ms, "full_attention_tflops": full_flops / (full_ms * 1e-3) / 1e12,
            "attention_time_ratio_full_over_pruned": full_ms / pruned_attn_ms}


def paper_form(path, torch, flush, steps):
    """The paper's exact gate form on the bench batch: score normalisation (Eq. (3)) over the
    step's scores, and Eq. (8) attention with the Eq. (7) temperature over the kept rows."""
    from learned_token_pruning_07_b300 import binding as tg
    wl = path.wl
    b_all = torch.empty_like(path.s)
    rng = np.random.default_rng(wl.seed + 5)
    gain = rng.uniform(0.5, 1.5, wl.H_q).astype(np.float32)
    temp = rng.uniform(0.8, 1.2, wl.H_q).astype(np.float32)
    d = path.d

    def norm():
        tg.normalize_scores(path.s, d["cu"], b_all, instr_mask=d["mask"], status=path.status)

    def attn():
        tg.gated_attention_eq8(d["Q"], d["K"], d["V"], path.cu_kept, path.pos_kept[:path.M], gain, temp, path.O,
                               max_seqlen=path.max_seqlen, b=path.g_kept[:path.M], status=path.status)

    def timed(fn):
        return graph_timed(fn, max(3, min(steps, 20)), torch, flush, 1000.0)

    # LN_2 fused into scoring: the bench's h stands for the raw residual a^L
    ln_w = torch.from_numpy(np.ascontiguousarray(
        rng.uniform(0.5, 1.5, wl.d).astype(np.float32))).to(torch.bfloat16).cuda().view(torch.int16)
    W1f = torch.empty_like(path.W1)
    tg.fold_rmsnorm_weight(path.W1, ln_w, W1f)

    def score_plain():
        tg.gate_score(d["h"], path.W1, path.w2, path.s, path.g, instr_mask=d["mask"], status=path.status)

    def score_norm():
        tg.gate_score_rmsnorm(d["h"], W1f, path.w2, path.s, path.g, instr_mask=d["mask"], status=path.status)

    norm_us, attn_us = timed(norm), timed(attn)
    plain_us, fused_us = timed(score_plain), timed(score_norm)
    assert tg.read_device_status(path.status) == 0, "device reported an error"
    flops = stage_work(wl, path.K, path.kept_lens)["gated_attention"]["flops"]
    return {"normalize_scores_us": norm_us, "attention_eq8_us": attn_us,
            "attention_eq8_tflops": flops / (attn_us * 1e-6) / 1e12,
            "gate_score_us": plain_us, "gate_score_rmsnorm_us": fused_us,
            "note": "each call captured in a CUDA graph and replayed between events after an L2 flush (median)"}


def two_budget(path, torch, flush, steps):
    """The packed two-budget forward (Eq. (9)) on the bench batch: one scoring pass, the full
    and the pruned keep lists packed as 2B sequences, then ONE attention call over the pack;
    against the same two budgets run as separate prune + attention calls."""
    from learned_token_pruning_07_b300 import binding as tg
    wl, T, B, d = path.wl, path.wl.T_total, path.wl.B, path.d
    e = lambda *shape, dt=torch.float32: torch.empty(*shape, dtype=dt, device="cuda")
    kept, cu = e(2 * T, dt=torch.int32), e(2 * B + 1, dt=torch.int32)
    h_kept, pos_kept, g_kept = e(2 * T, wl.d, dt=torch.int16), e(2 * T, dt=torch.int32), e(2 * T)
    M = T + path.M
    gen = torch.Generator(device="cuda").manual_seed(wl.seed + 9)
    Q = torch.randn((M, wl.H_q, wl.d_h), generator=gen, device="cuda").to(torch.bfloat16)
    Kt = torch.randn((M, wl.H_kv, wl.d_h), generator=gen, device="cuda").to(torch.bfloat16)
    V = torch.randn((M, wl.H_kv, wl.d_h), generator=gen, device="cuda").to(torch.bfloat16)
    O = torch.empty_like(Q)
    max_len = max(wl.seq_lens)

    def packed():
        tg.two_budget_prune_layer(d["h"], d["cu"], path.W1, path.w2, path.K, path.s, path.g, kept, cu, h_kept,
                                  pos_kept=pos_kept, g_kept=g_kept, pos=d["pos"], instr_mask=d["mask"],
                                  status=path.status)
        tg.gated_attention(Q, Kt, V, cu, path.tau, path.beta, O, max_seqlen=max_len, g=g_kept, status=path.status)

    def separate():
        path.step()   # the pruned budget: score, select, gather, attention
        tg.gated_attention(Q[:T], Kt[:T], V[:T], d["cu"], path.tau, path.beta, O[:T], max_seqlen=max_len,
                           g=path.g, status=path.status)  # the full budget's attention

    def timed(fn):
        return graph_timed(fn, max(3, min(steps, 10)), torch, flush, 1.0)

    p_ms, s_ms = timed(packed), timed(separate)
    assert tg.read_device_status(path.status) == 0, "device reported an error"
    del Q, Kt, V, O, h_kept
    torch.cuda.empty_cache()
    return {"K_full": "all document tokens", "K_prune": path.K, "packed_rows": M,
            "packed_ms": p_ms, "separate_ms": s_ms,
            "note": "one scoring pass + one attention call over the 2B-sequence pack, vs the pruned step plus "
                    "a separate full-budget attention call; each captured in a CUDA graph, replayed after an L2 flush"}


def backward(path, torch, flush, steps):
    """Next-row backward on the bench batch's kept rows: the forward with its log-sum-exp,
    the attention backward (dQ, dK, dV and the bias gradient, fp32 CUDA-core kernels) and
    the chain to the gate scores. Algorithmic FLOPs of the backward: 10 d_h per visible
    (query, key) pair per query head (S = QK^T recomputed once, dV, dP, dQ, dK)."""
    from learned_token_pruning_07_b300 import binding as tg
    wl, d, M = path.wl, path.d, path.M
    path.step()  # fills cu_kept, kept, g_kept for this batch
    e = lambda *shape, dt=torch.float32: torch.empty(*shape, dtype=dt, device="cuda")
    gen = torch.Generator(device="cuda").manual_seed(wl.seed + 11)
    dO = torch.randn((M, wl.H_q, wl.d_h), generator=gen, device="cuda").to(torch.bfloat16).view(torch.int16)
    lse = e(M, wl.H_q)
    dQ, dK, dV = e(M, wl.H_q, wl.d_h), e(M, wl.H_kv, wl.d_h), e(M, wl.H_kv, wl.d_h)
    dbias, ds = e(M, wl.H_q), e(wl.T_total)
    g_kept = path.g_kept[:M]

    def fwd():
        tg.gated_attention_lse(d["Q"], d["K"], d["V"], path.cu_kept, path.tau, path.beta, path.O, lse,
                               max_seqlen=path.max_seqlen, g=g_kept, status=path.status)

    def bwd():
        tg.gated_attention_bwd(d["Q"], d["K"], d["V"], path.O, dO, lse, path.cu_kept, path.tau, path.beta,
                               dQ, dK, dV, dbias, max_seqlen=path.max_seqlen, g=g_kept, status=path.status)

    def chain():
        tg.gate_score_grad(dbias, path.beta, g_kept, path.kept[:M], path.cu_kept, ds)

    def timed(fn):
        return graph_timed(fn, max(3, min(steps, 10)), torch, flush, 1000.0)

    f_us, b_us, c_us = timed(fwd), timed(bwd), timed(chain)
    assert tg.read_device_status(path.status) == 0, "device reported an error"
    pairs = sum(n * (n + 1) // 2 for n in path.kept_lens)
    bwd_flops = 10.0 * wl.d_h * wl.H_q * pairs
    del dO, lse, dQ, dK, dV, dbias, ds
    torch.cuda.empty_cache()
    return {"forward_lse_us": f_us, "attention_bwd_us": b_us, "gate_score_grad_us": c_us,
            "attention_bwd_tflops": bwd_flops / (b_us * 1e-6) / 1e12,
            "note": "tensor-core backward (row dots, dK/dV pass, dQ pass); each call captured in a CUDA graph and "
                    "replayed between events after an L2 flush (median)"}


def heads(path, torch, flush, steps):
    """Per-head gates on the bench batch: scoring with H_g = 16 gate heads (per-head scores and
    gates plus the head mean that selection ranks) against the single-gate score, and the
    attention with one gate column per query head against the shared gate."""
    from learned_token_pruning_07_b300 import binding as tg
    from learned_token_pruning_07_b300 import inputs as I
    wl, d, T, H_g = path.wl, path.d, path.wl.T_total, path.wl.H_q
    hw = I.make_gate_head_weights(wl, H_g)
    W2 = torch.from_numpy(hw["W2"].view(np.int16)).cuda()
    e = lambda *shape: torch.empty(*shape, dtype=torch.float32, device="cuda")
    s_h, g_h, sel = e(T, H_g), e(T, H_g), e(T)
    G = torch.from_numpy(I.make_head_gates(wl, path.M, H_g)).cuda()

    def score_heads():
        tg.gate_score_heads(d["h"], path.W1, W2, s_h, sel, g_heads=g_h, instr_mask=d["mask"], b2=hw["b2"],
                            status=path.status)

    def score_one():
        tg.gate_score(d["h"], path.W1, path.w2, path.s, path.g, instr_mask=d["mask"], status=path.status)

    def attn_heads():
        tg.gated_attention(d["Q"], d["K"], d["V"], path.cu_kept, path.tau, path.beta, path.O,
                           max_seqlen=path.max_seqlen, g=G, status=path.status)

    def attn_one():
        tg.gated_attention(d["Q"], d["K"], d["V"], path.cu_kept, path.tau, path.beta, path.O,
                           max_seqlen=path.max_seqlen, g=path.g_kept, status=path.status)

    def timed(fn):
        return graph_timed(fn, max(3, min(steps, 20)), torch, flush, 1000.0)

    path.step()  # cu_kept and g_kept for the kept rows
    out = {"H_g": H_g, "gate_score_heads_us": timed(score_heads), "gate_score_us": timed(score_one),
           "attention_per_head_gates_us": timed(attn_heads), "attention_shared_gate_us": timed(attn_one),
           "note": "each call captured in a CUDA graph and replayed between events after an L2 flush (median)"}
    assert tg.read_device_status(path.status) == 0, "device reported an error"
    return out


STAGE_NAMES = ["gate_score", "topk_select", "gather_kept", "gated_attention"]


def stage_summary(work, per_stage, peaks):
    """Per-kernel mean time and roofline fraction from the staged graph's event times (ms)."""
    stages = {}
    for i, n in enumerate(STAGE_NAMES):
        us = float(per_stage[:, i].mean()) * 1000.0
        w = work[n]
        if w["bound"] == "tensor":
            ach = w["flops"] / (us * 1e-6) / 1e12
            stages[n] = {"us": us, "bound": "tensor", "achieved_tflops": ach, "frac": ach / peaks["bf16_tflops"],
                         "achieved_gbs": w["bytes"] / (us * 1e-6) / 1e9}
        else:
            ach = w["bytes"] / (us * 1e-6) / 1e9
            stages[n] = {"us": us, "bound": "hbm", "achieved_gbs": ach, "frac": ach / peaks["hbm_gbs"]}
    return stages


def select_gather_summary(work, stages, peaks, paired_ms=None):
    """Selection and gather together against HBM: selection alone moves too few bytes to mean
    anything against HBM bandwidth. `us` / `frac` add the two staged kernel times; `paired_*`
    time the pair back to back with no event between them, as the fused call runs it."""
    us = stages["topk_select"]["us"] + stages["gather_kept"]["us"]
    by = work["topk_select"]["bytes"] + work["gather_kept"]["bytes"]
    out = {"us": us, "bytes": by, "achieved_gbs": by / (us * 1e-6) / 1e9,
           "frac": by / (us * 1e-6) / 1e9 / peaks["hbm_gbs"]}
    if paired_ms is not None:
        pu = float(paired_ms) * 1000.0
        out.update({"paired_us": pu, "paired_achieved_gbs": by / (pu * 1e-6) / 1e9,
                    "paired_frac": by / (pu * 1e-6) / 1e9 / peaks["hbm_gbs"]})
    return out


def other_configs(torch, flush, steps, peaks, rank, with_oracle=True):
    """Throughput lines of the other single-GPU workloads: the Qwen3-1.7B-shaped 8K gate layer
    (K = 1024) and the ragged batch of eight sequences (K = 2048 each, selection on 256-level
    scores), each with its per-kernel times and roofline fractions."""
    from learned_token_pruning_07_b300 import inputs as I
    out = []
    for name in ("qwen3_1p7b_8k", "ragged_b8"):
        base = I.WORKLOADS[name]
        wl = I.with_changes(base, seed=replica_seed(base.seed, rank))
        p = GatedPrefill(wl, wl.K, torch)
        g = GraphStep(p, torch)
        warm(g, 3, torch, flush)
        ps, pst = time_device_steps(g, max(5, min(steps, 30)), torch, flush)
        pair = time_pairs(g, max(5, min(steps, 30)), torch, flush)
        assert p.tg.read_device_status(p.status) == 0, "device reported an error"
        work = stage_work(wl, wl.K, p.kept_lens)
        st = stage_summary(work, pst, peaks)
        ms = float(ps.mean())
        entry = {"workload": workload_label(base, wl.K), "K": wl.K, "T_total": wl.T_total, "M_kept": p.M,
                 "value": wl.T_total / (ms / 1000.0), "unit": UNIT, "ms_per_step": ms, "stages": st,
                 "select_plus_gather": select_gather_summary(work, st, peaks, float(pair.mean())),
                 "selection_scores": ("synthetic 256-level quantised buffer" if wl.score_levels
                                      else "the step's own gate scores")}
        del g, p
        torch.cuda.empty_cache()
        if with_oracle:
            # one whole, unsampled oracle step of the same workload on the host cores
            t = oracle_step(base, base.K, {})
            entry["cpu_oracle"] = {"value": base.T_total / t["step"], "unit": UNIT, "ms_per_step": 1000.0 * t["step"],
                                   "stage_ms": {k: 1000.0 * v for k, v in t.items()}, "cores": blas_threads(),
                                   "kind": "oracle", "sample": oracle_sample_text(1, t["step"])}
        out.append(entry)
    return out


TIMING_NOTE = ("step captured in a CUDA graph (events only around the step, kernels chained by programmatic "
               "dependent launch); per-kernel times from a second graph with events between the kernels, on the "
               "launching stream; mean over steps; max over ranks")


def config_dict(wl, K, world):
    """The workload's description, the same in the GPU line and in the reference arm's line."""
    M = sum(min(K, a) + b for a, b in zip(wl.doc_lens, wl.instr_lens))
    return {"workload": workload_label(wl, K), "K": K, "T_total": wl.T_total, "M_kept": M,
            "parallelism": f"replicas x{world} (independent batches, no collective)", "l2": L2_NOTE,
            "timing": TIMING_NOTE}


def workload_label(wl, K):
    docs = wl.doc_lens if wl.B > 1 else wl.doc_lens[0]
    ins = wl.instr_lens if wl.B > 1 else wl.instr_lens[0]
    return (f"{wl.name}: B={wl.B}, doc={docs} + instr={ins} tokens, d={wl.d}, gate MLP {wl.d}->{wl.d_g}->1, "
            f"H_q={wl.H_q}, H_kv={wl.H_kv}, d_h={wl.d_h}, K={K}")


def run_reference(args, rank, world):
    """The reference arm: the oracle, timed on whole unsampled steps of the same workload on the
    host cores (rank 0 only; other ranks exit without work)."""
    from learned_token_pruning_07_b300 import inputs as I
    if rank != 0:
        return 0
    wl = I.WORKLOADS[args.workload]
    K = args.k if args.k is not None else wl.K
    cache = {}
    for _ in range(args.warmup):
        oracle_step(wl, K, cache)
    steps = [oracle_step(wl, K, cache) for _ in range(args.steps)]
    spent = sum(t["step"] for t in steps)
    ms = 1000.0 * spent / len(steps)
    value = wl.T_total / (ms / 1000.0)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(wl, K, world),
            "stage_ms": {k: 1000.0 * sum(t[k] for t in steps) / len(steps) for k in steps[0]},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
                             "sample": oracle_sample_text(len(steps), spent)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_gpu(args, rank, world, local):
    import torch
    from learned_token_pruning_07_b300 import build
    from learned_token_pruning_07_b300 import inputs as I
    build.build()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    base = I.WORKLOADS[args.workload]
    K = args.k if args.k is not None else base.K
    wl = I.with_changes(base, seed=replica_seed(base.seed, rank))
    path = GatedPrefill(wl, K, torch)
    flush = L2Flush(torch)
    torch.cuda.synchronize()

    # correctness gate before timing: the device status word must stay clean
    path.step()
    torch.cuda.synchronize()
    assert path.tg.read_device_status(path.status) == 0, "device reported an error"

    clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    gstep = GraphStep(path, torch)
    warm(gstep, args.warmup, torch, flush)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    per_step = time_whole_steps(gstep, args.steps, torch, flush)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    wall = time.perf_counter() - t_wall0
    per_stage = time_stages(gstep, args.steps, torch, flush)
    per_pair = time_pairs(gstep, args.steps, torch, flush)
    # keep the GPU busy a little longer so the sampler sees the clocks under this load
    t_end = time.perf_counter() + max(0.0, 1.0 - wall)
    while time.perf_counter() < t_end:
        gstep.replay()
        flush()
        torch.cuda.synchronize()
    clk = clocks.stop() if clocks else None
    assert path.tg.read_device_status(path.status) == 0, "device reported an error"

    ms_step = float(per_step.mean())
    ms_max = reduce_max(ms_step, world)
    value = aggregate(wl.T_total, world, ms_max / 1000.0)

    e2e_ms = reduce_max(float(time_e2e(path, max(3, min(args.steps, 20)), 2, torch).mean()), world)
    e2e_value = aggregate(wl.T_total, world, e2e_ms / 1000.0)

    peaks = load_peaks()
    work = stage_work(wl, K, path.kept_lens)
    names = STAGE_NAMES
    stages = stage_summary(work, per_stage, peaks)
    dom = max(names, key=lambda n: stages[n]["us"])
    w = work[dom]
    traffic = measured_traffic(dom, wl.name, K)
    if w["bound"] == "tensor":
        roof = {"kernel": dom, "bound": "tensor", "achieved": stages[dom]["achieved_tflops"],
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": stages[dom]["frac"], "traffic": traffic,
                "peak_source": f"{peaks['source']} bf16 dense (burst: the kernel is timed in a sub-ms step)"}
    else:
        roof = {"kernel": dom, "bound": "hbm", "achieved": stages[dom]["achieved_gbs"], "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": stages[dom]["frac"], "traffic": traffic,
                "peak_source": f"{peaks['source']} HBM copy bandwidth"}

    sweep = []
    if args.sweep and base.budgets and rank == 0:
        for Kb in base.budgets:
            p2 = path if Kb == K else GatedPrefill(wl, Kb, torch)
            g2 = gstep if p2 is path else GraphStep(p2, torch)
            warm(g2, 3, torch, flush)
            ps, pst = time_device_steps(g2, max(5, min(args.steps, 30)), torch, flush)
            wk = stage_work(wl, Kb, p2.kept_lens)
            a_us = float(pst[:, 3].mean()) * 1000.0
            sweep.append({"K": Kb, "M_kept": p2.M, "ms_per_step": float(ps.mean()),
                          "value": wl.T_total / (float(ps.mean()) / 1000.0),
                          "attention_tflops": wk["gated_attention"]["flops"] / (a_us * 1e-6) / 1e12,
                          "stage_us": [float(x) * 1000.0 for x in pst.mean(axis=0)], "stage_names": STAGE_NAMES})
            if p2 is not path:
                del g2, p2
                torch.cuda.empty_cache()

    extras = rank == 0 and args.extras
    others = (other_configs(torch, flush, args.steps, peaks, rank, with_oracle=world == 1 and not args.no_cpu_baseline)
              if (rank == 0 and args.configs) else None)
    paper = paper_form(path, torch, flush, args.steps) if extras else None
    twob = two_budget(path, torch, flush, args.steps) if extras else None
    bwd = backward(path, torch, flush, args.steps) if extras else None
    hds = heads(path, torch, flush, args.steps) if extras else None
    longctx = long_context(torch, flush, args.steps) if (args.long_context and rank == 0) else None

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(base, K)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_dict(base, K, world),
            "roofline": roof,
            "stages": stages,
            "select_plus_gather": select_gather_summary(work, stages, peaks, float(per_pair.mean())),
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "ms_per_step": e2e_ms,
                    "h2d_bytes_per_step": path.h2d_bytes(), "d2h_bytes_per_step": path.d2h_bytes(),
                    "api": "tg_gate_prune_layer + tg_gated_attention with pinned host buffers"},
            "gpu_launches": 4 * (args.steps),
            "clocks": clk,
            "wall_s_timed_region": wall,
        }
        if sweep:
            line["sweep"] = sweep
        if others:
            line["configs"] = others
        if paper:
            line["paper_form"] = paper
        if twob:
            line["two_budget"] = twob
        if bwd:
            line["backward"] = bwd
        if hds:
            line["heads"] = hds
        if longctx:
            line["long_context"] = longctx
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="sweep_32k")
    ap.add_argument("--k", type=int, default=None)
    ap.add_argument("--sweep", action=argparse.BooleanOptionalAction, default=True)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--long-context", action=argparse.BooleanOptionalAction, default=True,
                    help="also time the 128K workload: pruned step vs full causal attention")
    ap.add_argument("--configs", action=argparse.BooleanOptionalAction, default=True,
                    help="also time the 8K gate layer and the ragged batch of eight sequences")
    ap.add_argument("--extras", action=argparse.BooleanOptionalAction, default=True,
                    help="also measure the paper form, the two-budget pack, the backward and per-head gates")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)
    return run_gpu(args, rank, world, local)


if __name__ == "__main__":
    sys.exit(main())
