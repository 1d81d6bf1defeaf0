#!/usr/bin/env python3
"""Benchmark of the drafter-head + verifier hot path on GB300.

One step is one speculative round of the Llama-3.1-8B-shaped workload
(d=4096, r=512, V=128256, M=8 sequences, gamma=6, greedy): gamma low-rank head
calls (each M rows -> M drafted tokens; the drafter backbone between them is
out of scope, so each call gets its own synthetic hidden states) followed by
one greedy verification of the M sequences.  value = drafted tokens/s
(gamma * M per step), whole job over all ranks.

Inputs are resident in HBM; W_up is rotated over gamma copies (one per head
call) so every weight read of the timed region comes from HBM, not L2.  The
step is captured in a CUDA graph and replayed; sampling draws come from the
library's Philox stream (seed, offset), so the rounds have no uniform inputs.
Per-kernel times come from a CUPTI timeline of replays of the same captured
graph (kernel start and end on the GPU clock, dependent launches overlapping
as in the timed region); the dominant kernel's roofline divides its
algorithmic bytes by its mean span there.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

The default line also carries a compact "workloads" entry per other
configuration (GPT-OSS-20B, Qwen3-30B-A3B and SpecVocab @ Qwen3-8B shapes).
--impl reference times the CPU oracle on the host cores: whole rounds of the
same workload.  Multi-GPU: replicas only (the round has no exchange step);
one process per GPU under torchrun, barrier + max-over-ranks timing.
"""
from __future__ import annotations

import argparse
import hashlib
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "drafter head+sample tokens/s at V=128K-201K; verify steps/s; % of HBM roofline"
UNIT = "drafted tokens/s"
NOMINAL_HBM_GBS = 8000.0   # the roofline figure the workload's target names (8 TB/s)
L2_BYTES = 129e6
WORKLOADS = {
    # name: (d, r, V, M, gamma, temperature)
    "llama8b": (4096, 512, 128256, 8, 6, 0.0),
    "gptoss20b": (2880, 360, 201088, 16, 6, 0.7),
    "qwen30b": (2048, 256, 151936, 256, 4, 1.0),
    # SpecVocab: r here is the router width d' (router W_down d' x d, W_vocab V x d')
    "specvocab8b": (4096, 256, 151936, 32, 6, 1.0),
}
SPECVOCAB_K = 2048
WORKLOAD_DESC = {
    "llama8b": "Llama-3.1-8B-shaped speculative round: 6 low-rank head calls (M=8) + greedy verify (B=8)",
    "gptoss20b": "GPT-OSS-20B-shaped speculative round: 6 low-rank head calls (M=16, T=0.7) + sampling verify (B=16)",
    "qwen30b": "Qwen3-30B-A3B-shaped speculative round: 1 low-rank head call (M=256, T=1) + sampling verify (B=64)",
    "specvocab8b": "Qwen3-8B-shaped SpecVocab round: 6 dynamic-vocabulary head calls (M=32, d'=256, k=2048, T=1) + sampling verify (B=32)",
}
SEED, OFFSET = 20261202, 0   # the rounds' Philox stream (key and first counter offset)


# ----------------------------------------------------------------- ranks ---
def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    return world, rank, local


def aggregate(units_local: float, seconds_local: float, world: int):
    """Whole-job (units, seconds): units summed over ranks, time = max over ranks."""
    if world <= 1:
        return units_local, seconds_local
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" \
        else torch.device("cpu")
    t = torch.tensor([seconds_local], dtype=torch.float64, device=dev)
    u = torch.tensor([units_local], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(u.item()), float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- clocks ---
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons every 200 ms."""
    Q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.lines = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-i", str(gpu_index), "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        inside = [p for ts, p in rows if t0 <= ts <= t1]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"],
                    "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        mx = [num(p[2]) for p in inside if num(p[2]) is not None]
        pw = [num(p[3]) for p in inside if num(p[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4)
                          if p[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "power_w_max": max(pw) if pw else None, "samples": len(inside)}


# ------------------------------------------------------------ workload -----
def make_inputs(name: str, seed: int, dev, lowrank: bool = False, head_ranks=None):
    """Seeded synthetic tensors on the device: bf16 weights N(0, 1/fan_in),
    hidden states N(0, 1), Zipf-like target logits (-1.1 ln rank over a random
    permutation + N(0, 0.25)), draft logits = target + N(0, 1).  Drafted
    tokens are the draft rows' argmax (greedy) or a draw from softmax(draft/T).

    lowrank (sampling workloads): the draft side is the head's own; the
    target rows of the drafted positions are its draft logits z W_up^T
    (computed here with torch, before timing) + N(0, 1), the bonus rows
    Zipf-like, and every head call uses the same W_up (one drafter).

    head_ranks (low-rank workloads): head call j uses its own pair W_down_j
    (r_j x d) and W_up_j (V x r_j), a rank per drafted position."""
    import torch
    d, r, V, M, gamma, T = WORKLOADS[name]
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    n_calls = gamma if name != "qwen30b" else 1
    n_copies = max(n_calls, 2)
    w_down = (torch.randn(r, d, generator=g, device=dev) / d ** 0.5).to(torch.bfloat16)
    # the low-rank head's W_up, or SpecVocab's router matrix W_vocab (V x d')
    w_ups = [(torch.randn(V, r, generator=g, device=dev) / r ** 0.5).to(torch.bfloat16)
             for _ in range(n_copies)]
    w_downs = None
    if head_ranks:
        w_downs = [(torch.randn(rj, d, generator=g, device=dev) / d ** 0.5).to(torch.bfloat16)
                   for rj in head_ranks]
        w_ups = [(torch.randn(V, rj, generator=g, device=dev) / rj ** 0.5).to(torch.bfloat16)
                 for rj in head_ranks]
        r = int(round(sum(head_ranks) / len(head_ranks)))  # mean rank: bytes per call on average
    # SpecVocab's full head U (V x d, 1.2 GB: one copy, each call gathers its own rows)
    u_full = ((torch.randn(V, d, generator=g, device=dev) / d ** 0.5).to(torch.bfloat16)
              if name == "specvocab8b" else None)
    hidden = [torch.randn(M, d, generator=g, device=dev).to(torch.bfloat16)
              for _ in range(n_calls)]
    B = {"qwen30b": 64}.get(name, M)
    ranks = torch.argsort(torch.rand(B * (gamma + 1), V, generator=g, device=dev), dim=1)
    target = (-1.1 * torch.log(ranks.float() + 1.0)
              + 0.5 * torch.randn(B * (gamma + 1), V, generator=g, device=dev))
    target = target.reshape(B, gamma + 1, V).contiguous()
    del ranks
    draft = (target[:, :gamma] + torch.randn(B, gamma, V, generator=g, device=dev)).contiguous()
    if T > 0:
        probs = torch.softmax(draft / T, dim=2).reshape(B * gamma, V)
        tokens = torch.multinomial(probs, 1, generator=g).reshape(B, gamma).to(torch.int32)
        del probs
    else:
        tokens = torch.argmax(draft, dim=2).to(torch.int32)
    if lowrank:
        # position-major rows j*B + b: gamma calls of B rows, or one call of gamma*B
        del draft, tokens
        z = torch.cat([(h.float() @ w_down.float().t()).to(torch.bfloat16) for h in hidden])
        dl = (z.float() @ w_ups[0].float().t()).reshape(gamma, B, V)
        target = target.clone()
        target[:, :gamma] = dl.transpose(0, 1) + torch.randn(B, gamma, V, generator=g, device=dev)
        del z, dl
        draft, tokens = None, None
    return dict(name=name, d=d, r=r, V=V, M=M, B=B, gamma=gamma, T=T, n_calls=n_calls,
                w_down=w_down, w_ups=w_ups, u_full=u_full, hidden=hidden,
                target=target, lowrank=lowrank, w_downs=w_downs, ranks=head_ranks,
                draft=draft if T > 0 else None, tokens=tokens)


class Round:
    """Preallocated outputs / workspaces and the step as a sequence of library
    calls on the current stream.  Head call j draws at Philox offset
    OFFSET + j, the verifier at OFFSET + n_calls."""

    def __init__(self, x, ss):
        import torch
        self.x, self.ss = x, ss
        dev = x["w_down"].device
        M, d, r, V, B, gamma = x["M"], x["d"], x["r"], x["V"], x["B"], x["gamma"]
        self.specvocab = x["u_full"] is not None
        r_max = max(x["ranks"]) if x.get("ranks") else r
        hw = (ss.specvocab_head_workspace_size(M, d, r, V, SPECVOCAB_K) if self.specvocab
              else ss.slimspec_head_workspace_size(M, d, r_max, V, ss.SS_BF16))
        self.head_ws = torch.empty(hw, dtype=torch.uint8, device=dev)
        self.ver_ws = torch.empty(max(256, ss.spec_verify_workspace_size(B, gamma, V, x["T"])),
                                  dtype=torch.uint8, device=dev)
        self.head_out = [{"tokens": torch.empty(M, dtype=torch.int32, device=dev)}
                         for _ in range(x["n_calls"])]
        self.ver_out = {"tokens": torch.empty(B, gamma + 1, dtype=torch.int32, device=dev),
                        "num_accepted": torch.empty(B, dtype=torch.int32, device=dev)}
        self.lowrank = x.get("lowrank", False)
        if self.lowrank:
            # the head calls' outputs, position-major, as the verifier reads them
            n = gamma * B
            self.lr = {"z": torch.empty(n, r, dtype=torch.bfloat16, device=dev),
                       "logprob": torch.empty(n, dtype=torch.float32, device=dev),
                       "lse": torch.empty(n, dtype=torch.float32, device=dev),
                       "row_max": torch.empty(n, dtype=torch.float32, device=dev),
                       "tokens": torch.empty(n, dtype=torch.int32, device=dev)}
            self.head_out = [{k: v[j * M:(j + 1) * M] for k, v in self.lr.items()}
                             for j in range(x["n_calls"])]
            self.ver_ws = torch.empty(ss.spec_verify_lowrank_workspace_size(B, gamma, V, r),
                                      dtype=torch.uint8, device=dev)

    def head_call(self, j, hidden):
        """Head call j of the round (the low-rank head or the SpecVocab head)."""
        x, ss = self.x, self.ss
        T = x["T"]
        if self.specvocab:
            return ss.specvocab_head_forward(hidden, x["w_down"], x["w_ups"][j % len(x["w_ups"])],
                                             x["u_full"], SPECVOCAB_K, T, None, seed=SEED,
                                             offset=OFFSET + j, want_topk=False,
                                             workspace=self.head_ws, out=self.head_out[j])
        if self.lowrank:
            return ss.slimspec_head_forward(hidden, x["w_down"], x["w_ups"][0], T, None,
                                            seed=SEED, offset=OFFSET + j, want_stats=True,
                                            want_z=True, workspace=self.head_ws,
                                            out=self.head_out[j])
        w_down = x["w_downs"][j] if x.get("w_downs") else x["w_down"]
        return ss.slimspec_head_forward(hidden, w_down, x["w_ups"][j % len(x["w_ups"])], T, None,
                                        seed=SEED, offset=OFFSET + j, want_stats=False,
                                        workspace=self.head_ws, out=self.head_out[j])

    def verify(self, target, draft=None, tokens=None, out=None, lazy=False):
        x, ss = self.x, self.ss
        T, off = x["T"], OFFSET + x["n_calls"]
        out = out if out is not None else self.ver_out
        if self.lowrank:
            lr = self.lr
            return ss.spec_verify_lowrank(target, lr["z"], x["w_ups"][0], lr["logprob"],
                                          lr["lse"], lr["tokens"], T, None, seed=SEED,
                                          offset=off, position_major=True,
                                          workspace=self.ver_ws, out=out)
        return ss.spec_verify(target, draft, tokens, T, None, seed=SEED, offset=off, lazy=lazy,
                              workspace=self.ver_ws, out=out)

    def step(self):
        x = self.x
        for j in range(x["n_calls"]):
            self.head_call(j, x["hidden"][j])
        self.verify(x["target"], x["draft"], x["tokens"])


# ---------------------------------------------------------- byte counts ---
def head_stream_bytes(x) -> float:
    """Algorithmic bytes of one up-projection launch (k_head_stream or
    k_head_mma): the W_up stream (V*r*2) and the bf16 z rows it multiplies
    (M*r*2).  Partials are overhead."""
    M, r, V = x["M"], x["r"], x["V"]
    return V * r * 2 + M * r * 2


def head_call_bytes(x) -> float:
    """Algorithmic bytes of one whole head call: W_up + W_down + the hidden
    rows + the outputs (tokens, and the statistics and z when requested)."""
    M, d, r, V = x["M"], x["d"], x["r"], x["V"]
    out = M * 4 + (M * (3 * 4 + r * 2) if x.get("lowrank") else 0)
    return V * r * 2 + r * d * 2 + M * d * 2 + out


def verify_all_bytes(x) -> float:
    """Algorithmic bytes of one verification: every target row, plus every
    draft row when sampling with draft logits (the low-rank form reads W_up
    once instead), plus the drafted tokens."""
    B, g, V = x["B"], x["gamma"], x["V"]
    n = B * (g + 1) * V * 4 + B * g * 4
    if x["T"] > 0:
        n += B * g * V * 4 if not x.get("lowrank") else V * x["r"] * 2
    return n


def verify_rows_read(x, num_accepted) -> int:
    """Rows the accept chain needs: the target rows of positions 0..n_b of
    each sequence (n_b accepted), and when sampling the draft rows of the
    drafted positions among them.  The row pass reads at least these."""
    n = num_accepted.to("cpu").long()
    rows = int((n + 1).sum())
    if x["T"] > 0 and not x.get("lowrank", False):
        rows += int((n + 1).clamp(max=x["gamma"]).sum())
    return rows


def kernel_bytes(x, union_rows: float, ver_rows: int) -> dict:
    """Algorithmic bytes of one launch of each hot kernel (what the step must
    move at least once; partials and workspaces are overhead)."""
    M, d, r, V = x["M"], x["d"], x["r"], x["V"]
    out = {"k_head_mma": head_stream_bytes(x), "k_head_stream": head_stream_bytes(x),
           "k_down_proj": r * d * 2 + M * d * 2 + M * r * 2,
           "k_verify_rows": ver_rows * V * 4}
    if x["u_full"] is not None:
        out["k_gather_logits"] = union_rows * d * 2 + M * d * 2
        out["k_topk"] = M * V * 4
    return out


def specvocab_union_rows(x, rnd, ss) -> float:
    """Mean number of distinct U rows one SpecVocab call gathers (the union of
    its rows' top-k sets)."""
    import torch
    if x["u_full"] is None:
        return 0.0
    sizes = []
    for j in range(x["n_calls"]):
        o = ss.specvocab_head_forward(x["hidden"][j], x["w_down"], x["w_ups"][j % len(x["w_ups"])],
                                      x["u_full"], SPECVOCAB_K, x["T"], None, seed=SEED,
                                      offset=OFFSET + j, want_topk=True, workspace=rnd.head_ws)
        sizes.append(torch.unique(o["topk_idx"]).numel())
    return float(sum(sizes)) / len(sizes)


def profiled_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes from the committed ncu summary of this kernel, or
    None when there is none or the kernel source changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.txt")
    if not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if ":" in line:
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    src_file = {"k_head_mma": "head_mma.cu", "k_head_stream": "head.cu", "k_down_proj": "head.cu",
                "k_verify_rows": "verify.cu", "k_topk": "specvocab.cu",
                "k_gather_logits": "specvocab.cu"}.get(kernel)
    if src_file is None:
        return None
    src = os.path.join(ROOT, "speculative_decoding_drafter_slimspec_gb300", "csrc", src_file)
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    if fields.get("source_sha256") != sha:
        return None
    try:
        return float(fields["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def measured_tensor_peak():
    """Dense bf16 tensor peak (TFLOP/s): the measured burst figure, else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        return float(json.load(open(path))["bf16_tflops"])
    return 1900.0


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def hbm_roofline(kernel, nbytes, seconds, peak, peak_kind, workload=None) -> dict:
    ach = nbytes / seconds / 1e9
    return {"kernel": kernel, "bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s",
            "frac": ach / peak, "frac_of_8tbs": ach / NOMINAL_HBM_GBS,
            "traffic": profiled_traffic(kernel, workload) if workload else None,
            "algorithmic_bytes_per_launch": nbytes, "peak_source": peak_kind,
            "us_per_launch": seconds * 1e6}


# ------------------------------------------------------- timeline / timing --
def graph_timeline(graph, stream, n, launches_per_step) -> dict | None:
    """Per-kernel figures from a CUPTI timeline of n replays of the captured
    step (speculative_decoding_drafter_slimspec_gb300.timeline)."""
    import torch
    from speculative_decoding_drafter_slimspec_gb300 import timeline
    if not timeline.available():
        return None
    with timeline.KernelTimeline() as tl:
        with torch.cuda.stream(stream):
            for _ in range(n):
                graph.replay()
        stream.synchronize()
    return timeline.summarize(tl.records, launches_per_step)


def head_call_period(tsum, n_calls) -> dict | None:
    """Head-call time in the replayed round, from the timeline: the head phase
    (first library kernel's start to the last head kernel's end) per call,
    and the steady period between the ends of consecutive calls' last
    kernels (calls 1..n-1)."""
    if not tsum or not tsum.get("replay_records"):
        return None
    head_kinds = ("k_head_mma_finish", "k_head_stream", "k_cand_finish")
    phases, periods = [], []
    for grp in tsum["replay_records"]:
        ends = [e for kind, _, e in grp if kind in head_kinds]
        if len(ends) < n_calls:   # a head without a separate finish launch
            ends = [e for kind, _, e in grp if kind == "k_head_mma"]
        if len(ends) < n_calls:
            return None
        ends = sorted(ends)[:n_calls]
        phases.append((ends[-1] - grp[0][1]) / n_calls)
        periods += [b - a for a, b in zip(ends[:-1], ends[1:])]
    return {"us_per_call": statistics.mean(phases) / 1e3,
            "steady_us_per_call": statistics.mean(periods) / 1e3 if periods else None,
            "how": "CUPTI timeline of the replayed round: head phase per call (first kernel's "
                   "start to the last call's end), and the period between consecutive calls' ends"}


def verify_phase(tsum) -> float | None:
    """Time of the verification in the replayed round, in us: from its first
    kernel's start (or the end of the drafting kernels before it, if it
    started early as a dependent launch) to the round's last end."""
    if not tsum or not tsum.get("replay_records"):
        return None
    out = []
    for grp in tsum["replay_records"]:
        first = next((i for i, (kind, _, _) in enumerate(grp) if kind.startswith("k_verify")),
                     None)
        if first is None:
            return None
        start = grp[first][1]
        if first > 0:
            start = max(start, max(e for _, _, e in grp[:first]))
        out.append(max(e for _, _, e in grp) - start)
    return statistics.mean(out) / 1e3


def quantiles(values, fracs):
    """Nearest-rank quantiles of a list of numbers."""
    v = sorted(values)
    return [v[min(len(v) - 1, int(f * (len(v) - 1) + 0.5))] for f in fracs]


def step_time_distribution(graph, stream, n):
    """p10 / median / p90 of the step time over n more replays of the captured
    step, each between its own pair of CUDA events (taken after the timed
    region, which has only one pair; the events add a little to each step)."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    with torch.cuda.stream(stream):
        for a, b in evs:
            a.record(stream)
            graph.replay()
            b.record(stream)
    stream.synchronize()
    p10, p50, p90 = quantiles([a.elapsed_time(b) for a, b in evs], (0.1, 0.5, 0.9))
    return {"p10": p10, "median": p50, "p90": p90, "steps": n,
            "how": "an event pair around each replay, after the timed region"}


def clock_window(graph, stream, seconds: float, step_ms: float) -> dict:
    """Replays the step for `seconds` right after the timed region, so that a
    200 ms nvidia-smi sampler (running since before the timed region) sees
    the GPU under this load; returns the window's replays and step time."""
    import torch
    n = max(10, int(seconds * 1000.0 / max(step_ms, 1e-3)))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(n):
            graph.replay()
        e1.record(stream)
    stream.synchronize()
    return {"replays": n, "seconds": time.time() - t0, "ms_per_step": e0.elapsed_time(e1) / n,
            "how": "replays right after the timed region, sampled every 200 ms"}


def timed_verify(x, rnd, ss, stream, steps, lazy=False) -> dict:
    """spec_verify (or spec_verify_lowrank) alone: a graph of one call per
    copy of the target (and draft) rows, enough copies that the rows read
    between two reads of one copy exceed L2; steps/s = calls / time.  lazy:
    the position-by-position schedule (spec_verify_lazy) instead."""
    import torch
    per_copy = x["B"] * (x["gamma"] + 1) * x["V"] * 4 + (
        x["B"] * x["gamma"] * x["V"] * 4 if x["draft"] is not None else 0)
    n_copies = max(2, int(math.ceil(2 * L2_BYTES / per_copy)) + 1)
    tg = [x["target"]] + [x["target"].clone() for _ in range(n_copies - 1)]
    dr = ([x["draft"]] + [x["draft"].clone() for _ in range(n_copies - 1)]
          if x["draft"] is not None else [None] * n_copies)
    with torch.cuda.stream(stream):
        for i in range(n_copies):
            rnd.verify(tg[i], dr[i], x["tokens"], lazy=lazy)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
        for i in range(n_copies):
            rnd.verify(tg[i], dr[i], x["tokens"], lazy=lazy)
    reps = max(3, steps // n_copies + 1)
    with torch.cuda.stream(stream):
        for _ in range(3):
            graph.replay()
    stream.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            graph.replay()
        e1.record(stream)
    stream.synchronize()
    us = e0.elapsed_time(e1) * 1000.0 / (reps * n_copies)
    del tg, dr, graph
    return {"us_per_call": us, "steps_per_s": 1e6 / us, "calls": reps * n_copies,
            "input_copies": n_copies,
            "how": "CUDA graph of one verification per copy of the rows, replayed; events"}


# ------------------------------------------------------------ CPU oracle ---
def numpy_inputs(x):
    """The round's inputs as numpy arrays (fp32 values; bf16 weights exact)."""
    def f(t):
        return t.float().cpu().numpy() if t is not None else None
    return dict(name=x["name"], V=x["V"], M=x["M"], B=x["B"], gamma=x["gamma"], T=x["T"],
                n_calls=x["n_calls"], d=x["d"], r=x["r"],
                hidden=[f(h) for h in x["hidden"]], w_down=f(x["w_down"]),
                w_ups=[f(w) for w in x["w_ups"][:x["n_calls"]]],
                target=f(x["target"]), draft=f(x["draft"]),
                tokens=x["tokens"].cpu().numpy() if x["tokens"] is not None else None,
                u_full=f(x["u_full"]))


def oracle_round(x_np):
    """One whole round through the CPU oracle: every head call (all M rows over
    the full vocabulary) and the verification of all B sequences, drawing the
    Philox uniforms the library draws."""
    import oracle
    T, M, B, g = x_np["T"], x_np["M"], x_np["B"], x_np["gamma"]
    for j in range(x_np["n_calls"]):
        u = oracle.philox_uniforms(SEED, OFFSET + j, M, 1)[:, 0] if T > 0 else None
        w_up = x_np["w_ups"][j % len(x_np["w_ups"])]
        if x_np.get("u_full") is not None:
            oracle.specvocab_head(x_np["hidden"][j], x_np["w_down"], w_up, x_np["u_full"],
                                  SPECVOCAB_K, T, u)
        else:
            oracle.slimspec_head(x_np["hidden"][j], x_np["w_down"], w_up, "bf16", T, u)
    uv = oracle.philox_uniforms(SEED, OFFSET + x_np["n_calls"], B, g + 1) if T > 0 else None
    oracle.verify_batch(x_np["target"], x_np["draft"], x_np["tokens"], uv, T)


def oracle_rate(x_np, budget_s: float, min_rounds: int = 1) -> dict:
    """Whole oracle rounds for about budget_s (at least min_rounds)."""
    units = x_np["n_calls"] * x_np["M"]
    times = []
    t_all = time.perf_counter()
    while len(times) < min_rounds or time.perf_counter() - t_all < budget_s:
        t0 = time.perf_counter()
        oracle_round(x_np)
        times.append(time.perf_counter() - t0)
    return {"value": units * len(times) / sum(times), "rounds": len(times),
            "seconds": sum(times), "round_s": statistics.mean(times)}


def single_thread_oracle(workload: str, rounds: int = 2):
    """The same oracle round on one host core: a child process whose BLAS
    thread counts are fixed to 1 before numpy loads.  It builds its own
    inputs of the workload's shapes (the oracle's cost does not depend on the
    values).  Returns drafted tokens/s, or None if the child failed."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1",
               NUMEXPR_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    code = ("import bench, json; "
            f"print(json.dumps(bench._child_single_thread({workload!r}, {rounds})))")
    try:
        r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                           text=True, timeout=900)
        return json.loads(r.stdout.strip().splitlines()[-1])
    except (subprocess.SubprocessError, ValueError, IndexError):
        return None


def _child_single_thread(workload: str, rounds: int) -> dict:
    import torch
    torch.set_num_threads(1)
    x = make_inputs(workload, 1234, torch.device("cpu"))
    r = oracle_rate(numpy_inputs(x), 0.0, min_rounds=rounds)
    r["cores"] = 1
    return r


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def config_dict(workload):
    d, r, V, M, gamma, T = WORKLOADS[workload]
    if workload == "specvocab8b":
        return {"workload": WORKLOAD_DESC[workload], "d": d, "d_prime": r, "V": V, "k": SPECVOCAB_K,
                "M": M, "gamma": gamma, "temperature": T, "parallelism": "replicas",
                "l2": "W_vocab rotated over one copy per head call, U (1.2 GB) and the gathered "
                      "rows (~0.4 GB per call) larger than L2"}
    return {"workload": WORKLOAD_DESC[workload], "d": d, "r": r, "V": V, "M": M,
            "gamma": gamma, "temperature": T, "parallelism": "replicas",
            "l2": "W_up rotated over one copy per head call and the round reads "
                  ">750 MB between re-reads; inputs larger than L2"}


# ----------------------------------------------------------------- arms ---
def run_reference(args, world, rank):
    """CPU oracle arm: rank 0 alone times K whole rounds (after W)."""
    if rank != 0:
        return
    import torch
    # inputs built on the CPU with the same recipe (no GPU needed for this arm)
    x = make_inputs(args.workload, 1234, torch.device("cpu"))
    x_np = numpy_inputs(x)
    t0 = time.perf_counter()
    oracle_round(x_np)                                 # the first warm-up round, timed for sizing
    t_round = time.perf_counter() - t0
    # whole rounds; as many of the K asked for as fit the run's budget
    budget = 170.0
    units = x["n_calls"] * x["M"]
    fit = max(1, int(budget / max(t_round, 1e-6)))
    warm = max(0, min(args.warmup - 1, fit // 4))
    for _ in range(warm):
        oracle_round(x_np)
    n = max(1, min(args.steps, fit - warm - 1))
    r = oracle_rate(x_np, 0.0, min_rounds=n)
    rate = r["value"]
    sample = (f"{n} whole rounds ({units} head rows over all {x['V']} vocabulary rows + "
              f"{x['B']} verified sequences each), {r['seconds']:.1f} s"
              + ("" if n == args.steps else f"; {args.steps} steps would exceed the run's budget"))
    line = {"impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * units / rate, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(args.workload),
            "cpu_baseline": {"value": rate, "unit": UNIT, "cores": cores(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def dense_head_comparison(x, head_us):
    """The dense V x d head the low-rank head replaces, as one cuBLAS bf16 GEMM
    (torch.matmul, logits only, no reduction) on the same GPU."""
    import torch
    dev = x["w_down"].device
    M, d, V = x["M"], x["d"], x["V"]
    g = torch.Generator(device=dev)
    g.manual_seed(99)
    w = (torch.randn(V, d, generator=g, device=dev) / d ** 0.5).to(torch.bfloat16)
    h = x["hidden"][0]
    for _ in range(3):
        torch.matmul(h, w.t())
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    n = 20
    e0.record()
    for _ in range(n):
        torch.matmul(h, w.t())
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1000.0 / n
    nbytes = V * d * 2
    del w
    return {"kernel": "cuBLAS bf16 GEMM via torch.matmul (dense V x d logits, no reduction)",
            "us_per_call": us, "bytes": nbytes, "GB/s": nbytes / us / 1e3,
            "low_rank_head_call_us": head_us,
            "speedup_vs_dense": (us / head_us) if head_us else None}


def trimmed_head_comparison(x, head_us, kept=32768):
    """The static trimmed head (FR-Spec / VocabTrim form) on the same GPU: the
    dense head over `kept` of the V vocabulary rows (d = 4096, bf16, the same
    M rows, greedy), through this library's tensor-core kernel, two copies of
    W_kept alternating so every call reads HBM."""
    import torch
    import speculative_decoding_drafter_slimspec_gb300 as ss
    dev = x["w_down"].device
    M, d, V = x["M"], x["d"], x["V"]
    g = torch.Generator(device=dev)
    g.manual_seed(98)
    ws = [(torch.randn(kept, d, generator=g, device=dev) / d ** 0.5).to(torch.bfloat16)
          for _ in range(2)]
    ids = torch.sort(torch.randperm(V, generator=g, device=dev)[:kept]).values.to(torch.int32)
    h = x["hidden"][0]
    wsp = torch.empty(ss.trimmed_head_workspace_size(M, d, kept), dtype=torch.uint8, device=dev)
    out = {"tokens": torch.empty(M, dtype=torch.int32, device=dev)}
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for j in range(4):
            ss.trimmed_head_forward(h, ws[j % 2], ids, 0.0, want_stats=False, workspace=wsp,
                                    out=out)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
            for j in range(10):
                ss.trimmed_head_forward(h, ws[j % 2], ids, 0.0, want_stats=False, workspace=wsp,
                                        out=out)
        for _ in range(3):
            graph.replay()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(20):
            graph.replay()
        e1.record(stream)
    stream.synchronize()
    us = e0.elapsed_time(e1) * 1000.0 / 200
    nbytes = kept * d * 2 + M * d * 2
    return {"kernel": "k_head_mma over the kept rows (z = h, K = d) + k_head_mma_finish",
            "kept_rows": kept, "us_per_call": us, "bytes": nbytes, "GB/s": nbytes / us / 1e3,
            "low_rank_head_call_us": head_us,
            "note": "the low-rank head scores all V rows; the trimmed head never drafts the "
                    f"{V - kept} dropped ids"}


def run_e2e(args, x, ss, stream, world):
    """The round through the Python API with pinned host inputs copied in and
    the tokens copied out inside the timed region, every step, in the order a
    live round has them: the drafting calls' hidden rows first, then the
    drafting calls, then the verifier's rows (a live target produces them only
    after drafting), the verification, and one device-to-host copy of every
    token.  All on the launching stream."""
    import torch
    dev = x["w_down"].device
    T, M, n_calls, B, gamma = x["T"], x["M"], x["n_calls"], x["B"], x["gamma"]
    lowrank = x.get("lowrank", False)
    h_host = torch.stack([h.cpu() for h in x["hidden"]]).pin_memory()
    h_dev = torch.empty_like(h_host, device=dev)
    # the verifier's host inputs: target rows always; draft rows and tokens
    # unless the draft side comes from the drafting calls
    v_host = {"target": x["target"].cpu().pin_memory()}
    if not lowrank:
        v_host["tokens"] = x["tokens"].cpu().pin_memory()
        if T > 0:
            v_host["draft"] = x["draft"].cpu().pin_memory()
    v_dev = {k: torch.empty_like(v, device=dev) for k, v in v_host.items()}

    # one result buffer: every call writes its tokens straight into it, so
    # the step has no device-to-device copy; each slot starts 16-byte aligned
    def pad4(k):
        return (k + 3) // 4 * 4
    n = B * (gamma + 1)
    slot = M if lowrank else pad4(M)  # the low-rank calls' rows stay contiguous
    off = pad4(n_calls * slot)
    out_host = torch.empty(off + pad4(n) + B, dtype=torch.int32).pin_memory()
    res = torch.empty_like(out_host, device=dev)
    rnd = Round(x, ss)
    if lowrank:
        rnd.lr["tokens"] = res[:n_calls * M]
        rnd.head_out = [{k: v[j * M:(j + 1) * M] for k, v in rnd.lr.items()}
                        for j in range(n_calls)]
    else:
        for j in range(n_calls):
            rnd.head_out[j]["tokens"] = res[j * slot:j * slot + M]
    ver_out = {"tokens": res[off:off + n].view(B, gamma + 1),
               "num_accepted": res[off + pad4(n):off + pad4(n) + B]}

    def step():
        h_dev.copy_(h_host, non_blocking=True)
        for j in range(n_calls):
            rnd.head_call(j, h_dev[j])
        for k in v_host:
            v_dev[k].copy_(v_host[k], non_blocking=True)
        rnd.verify(v_dev["target"], v_dev.get("draft"), v_dev.get("tokens"), out=ver_out)
        out_host.copy_(res, non_blocking=True)

    n_steps = min(args.steps, args.e2e_steps)

    def timed(run):
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(n_steps):
                run()
            e1.record(stream)
        stream.synchronize()
        barrier(world)
        return e0.elapsed_time(e1) / 1000.0

    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
    stream.synchronize()
    # the calls issued one by one from Python, every step
    eager_units, eager_secs = aggregate(n_calls * M * n_steps, timed(step), world)
    # the same calls, copies included, captured once and replayed every step
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
        step()
    with torch.cuda.stream(stream):
        for _ in range(3):
            graph.replay()
    stream.synchronize()
    sec_local = timed(graph.replay)
    units, secs = aggregate(n_calls * M * n_steps, sec_local, world)
    # the copied-in round must give the device-resident round's tokens
    ref = Round(x, ss)
    with torch.cuda.stream(stream):
        ref.step()
    stream.synchronize()
    got_v = out_host[off:off + n].reshape(B, gamma + 1)
    want = ref.ver_out["tokens"].cpu()
    acc = ref.ver_out["num_accepted"].cpu()
    for b in range(B):
        assert torch.equal(got_v[b, :acc[b] + 1], want[b, :acc[b] + 1]), "e2e tokens differ"
    assert torch.equal(out_host[off + pad4(n):off + pad4(n) + B], acc), \
        "e2e acceptance counts differ"
    for j in range(n_calls):
        s = j * slot
        assert torch.equal(out_host[s:s + M], ref.head_out[j]["tokens"].cpu()), \
            "e2e drafted tokens differ"
    h2d = h_host.numel() * h_host.element_size() + sum(
        v.numel() * v.element_size() for v in v_host.values())
    return {"value": units / secs, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(out_host.numel() * 4), "steps": n_steps,
            "issue": "the step's copies and calls captured once in a CUDA graph, replayed per step",
            "order": "hidden rows in, drafting calls, verifier rows in, verification, tokens out; "
                     "one stream",
            "eager_value": eager_units / eager_secs}


def measure_round(args, ss, dev, local, world, workload, lowrank=False, ranks=None,
                  full=True) -> dict:
    """Times one workload's round and returns its bench fields: value and
    step time (CUDA events around K replays of the captured step, max over
    ranks), the CUPTI per-kernel figures, rooflines, the verifier timed
    alone, and (full) the step time distribution, the clock window and e2e."""
    import torch
    rank = int(os.environ.get("RANK", "0"))
    x = make_inputs(workload, 1234 + rank, dev, lowrank=lowrank, head_ranks=ranks)
    rnd = Round(x, ss)
    stream = torch.cuda.Stream(device=dev)
    units_per_step = x["n_calls"] * x["M"]

    # warm-up eagerly (also sets kernel attributes before capture)
    with torch.cuda.stream(stream):
        for _ in range(3):
            rnd.step()
    stream.synchronize()
    assert ss.ss_get_device_error() == ss.SS_OK
    with torch.cuda.stream(stream):
        union_rows = specvocab_union_rows(x, rnd, ss)
    stream.synchronize()
    ver_rows = verify_rows_read(x, rnd.ver_out["num_accepted"])

    graph = torch.cuda.CUDAGraph()
    n0 = ss.launch_count()
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
        rnd.step()
    launches_per_step = ss.launch_count() - n0

    sampler = ClockSampler(local) if full and not args.no_clocks else None
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    stream.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        e1.record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    sec_local = e0.elapsed_time(e1) / 1000.0
    units, secs = aggregate(units_per_step * args.steps, sec_local, world)
    assert ss.ss_get_device_error() == ss.SS_OK
    ms_step = secs * 1000.0 / args.steps
    out = {"value": units / secs, "ms_per_step": ms_step,
           "gpu_launches": int(launches_per_step * args.steps),
           "launches_per_step": launches_per_step, "x": x}

    if sampler:
        # the timed region is milliseconds long: keep the GPU under the same
        # load for a window the sampler can see
        win = clock_window(graph, stream, args.clock_seconds, ms_step)
        time.sleep(0.3)
        sampler.stop()
        out["clocks"] = sampler.summary(wall0, time.time())
        out["clocks"]["window"] = win
    # per-kernel figures from the replayed step's CUPTI timeline
    tsum = None if args.no_timeline else \
        graph_timeline(graph, stream, max(10, min(50, args.steps)), launches_per_step)
    ver_in_round = verify_phase(tsum)
    peak, peak_kind = measured_peaks()
    kb = kernel_bytes(x, union_rows, ver_rows)
    roof = head_roof = call_roof = None
    kern = {}
    if tsum and tsum["kernels"]:
        kern = tsum["kernels"]
        if "k_verify_rows" in kern:
            # the row pass may be split in two launches: its bytes are per step
            kb["k_verify_rows"] /= kern["k_verify_rows"]["launches_per_step"]
        cands = [k for k in kern if k in kb]
        if cands:
            dom = max(cands, key=lambda k: kern[k]["exclusive_us_per_step"])
            roof = hbm_roofline(dom, kb[dom], kern[dom]["us_per_launch"] / 1e6, peak, peak_kind,
                                workload)
        hk = next((k for k in ("k_head_mma", "k_head_stream") if k in kern), None)
        if hk:
            head_roof = hbm_roofline(hk, kb[hk], kern[hk]["us_per_launch"] / 1e6, peak,
                                     peak_kind, workload)
            if hk == "k_head_mma":
                flops = 2.0 * x["M"] * x["V"] * x["r"]
                tpeak = measured_tensor_peak()
                dur = kern[hk]["us_per_launch"] / 1e6
                head_roof["tensor"] = {"achieved": flops / dur / 1e12, "peak": tpeak,
                                       "unit": "TFLOP/s", "frac": flops / dur / 1e12 / tpeak,
                                       "algorithmic_flops_per_launch": flops}
            if roof and roof["kernel"] == hk:
                roof = dict(head_roof)
        if x["u_full"] is None:
            hc = head_call_period(tsum, x["n_calls"])
            if hc:
                nb = head_call_bytes(x)
                call_roof = hbm_roofline("head call (all kernels)", nb, hc["us_per_call"] / 1e6,
                                         peak, peak_kind)
                call_roof.update(hc)
                if hc.get("steady_us_per_call"):
                    st = hbm_roofline("", nb, hc["steady_us_per_call"] / 1e6, peak, peak_kind)
                    call_roof["steady"] = {"achieved": st["achieved"], "frac": st["frac"],
                                           "frac_of_8tbs": st["frac_of_8tbs"]}
        tsum.pop("replay_records", None)
    out.update(roofline=roof, head_roofline=head_roof,
               head_call_roofline=call_roof, kernels=kern,
               timeline={k: v for k, v in (tsum or {}).items() if k != "kernels"},
               union_rows=union_rows)
    # the verifier alone
    vt = timed_verify(x, rnd, ss, stream, args.steps)
    vt["in_round_us"] = ver_in_round
    nb = verify_all_bytes(x)
    vr = hbm_roofline("verification (all kernels)", nb, vt["us_per_call"] / 1e6, peak, peak_kind)
    vt["roofline_all_rows"] = {k: vr[k] for k in ("achieved", "peak", "unit", "frac",
                                                  "frac_of_8tbs", "algorithmic_bytes_per_launch")}
    out["verify"] = vt
    # the rows the accept chain needs over the same time: how close the
    # verification comes to reading only those
    ver_roof = hbm_roofline("verification (all kernels, timed alone)", ver_rows * x["V"] * 4,
                            vt["us_per_call"] / 1e6, peak, peak_kind)
    ver_roof["rows_needed"] = ver_rows
    ver_roof["rows_total"] = x["B"] * (x["gamma"] + 1) + (
        x["B"] * x["gamma"] if x["T"] > 0 and not x.get("lowrank", False) else 0)
    if not x.get("lowrank", False):
        # the lazy schedule (spec_verify_lazy): exactly the needed rows, one
        # row pass and one decision per position
        vl = timed_verify(x, rnd, ss, stream, args.steps, lazy=True)
        lr = hbm_roofline("verification, lazy schedule (timed alone)", ver_rows * x["V"] * 4,
                          vl["us_per_call"] / 1e6, peak, peak_kind)
        ver_roof["lazy_schedule"] = {"us_per_call": vl["us_per_call"], "achieved": lr["achieved"],
                                     "frac": lr["frac"], "frac_of_8tbs": lr["frac_of_8tbs"]}
    out["verify_roofline"] = ver_roof
    if full:
        out["ms_per_step_dist"] = step_time_distribution(graph, stream, min(args.steps, 500))
    del graph
    if full and not args.no_e2e:
        out["e2e"] = run_e2e(args, x, ss, stream, world)
    return out


def line_from(meas, args, world, workload, lowrank=False, ranks=None) -> dict:
    x = meas["x"]
    line = {"metric": METRIC, "value": meas["value"], "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": meas["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic: seeded N(0,1/fan_in) bf16 weights, N(0,1) hidden states, "
                    "Zipf-like target logits; sampling draws from the Philox stream",
            "config": dict(config_dict(workload), **(
                {"verify": "draft side from the head calls (z, log q, lse; spec_verify_lowrank), "
                           "one W_up for all calls"} if lowrank else {}),
                **({"ranks_per_position": ranks} if ranks else {})),
            "roofline": meas["roofline"], "head_roofline": meas["head_roofline"],
            "head_call_roofline": meas["head_call_roofline"],
            "verify_roofline": meas["verify_roofline"], "verify": meas["verify"],
            "verify_steps_per_s": meas["verify"]["steps_per_s"],
            "specvocab_union_rows": meas["union_rows"] if x["u_full"] is not None else None,
            "gpu_launches": meas["gpu_launches"], "kernels": meas["kernels"],
            "kernel_timing": "CUPTI timeline of replays of the timed graph: us_per_launch = mean "
                             "span (start to end) of a launch; exclusive_us_per_step = busy time "
                             "first covered by the kernel's launches (sums to the busy time)",
            "timeline": meas["timeline"]}
    for k in ("ms_per_step_dist", "clocks", "e2e"):
        if k in meas:
            line[k] = meas[k]
    return line


def compact(meas) -> dict:
    """The fields of a workload kept in the default line's 'workloads' key."""
    keep = ("value", "ms_per_step", "gpu_launches")
    out = {k: meas[k] for k in keep}
    for k in ("roofline", "head_roofline", "head_call_roofline", "verify_roofline"):
        r = meas.get(k)
        if r:
            out[k] = {kk: r[kk] for kk in ("kernel", "achieved", "frac", "frac_of_8tbs",
                                           "us_per_launch", "traffic", "steady",
                                           "lazy_schedule")
                      if kk in r}
    v = meas["verify"]
    out["verify"] = {"us_per_call": v["us_per_call"], "steps_per_s": v["steps_per_s"],
                     "in_round_us": v.get("in_round_us"),
                     "roofline_all_rows_frac": v["roofline_all_rows"]["frac"]}
    out["kernels"] = {k: {"us_per_launch": round(kk["us_per_launch"], 3),
                          "share": round(kk["share"], 4)} for k, kk in meas["kernels"].items()}
    if meas.get("union_rows"):
        out["specvocab_union_rows"] = meas["union_rows"]
    if "e2e" in meas:
        out["e2e"] = {k: meas["e2e"][k] for k in ("value", "h2d_bytes_per_step",
                                                  "d2h_bytes_per_step", "eager_value")}
    return out


def run_ours(args, world, rank, local):
    import torch
    import speculative_decoding_drafter_slimspec_gb300 as ss
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lowrank = args.verify == "lowrank"
    if lowrank and (WORKLOADS[args.workload][5] <= 0 or args.workload == "specvocab8b"):
        raise SystemExit("--verify lowrank needs a sampling low-rank workload (gptoss20b, qwen30b)")
    ranks = [int(v) for v in args.ranks.split(",")] if args.ranks else None
    if ranks and (args.workload in ("specvocab8b", "qwen30b") or lowrank or
                  len(ranks) != WORKLOADS[args.workload][4]):
        raise SystemExit("--ranks needs one rank per head call of a low-rank workload "
                         "(gamma calls), without --verify lowrank")
    meas = measure_round(args, ss, dev, local, world, args.workload, lowrank, ranks, full=True)
    x = meas["x"]
    if rank != 0:
        return
    line = line_from(meas, args, world, args.workload, lowrank, ranks)
    call_us = (meas["head_call_roofline"] or {}).get("us_per_call")
    if args.workload == "llama8b" and not args.no_dense:
        # the Llama-shaped configuration also names the dense 128256 x 4096 head
        line["dense_head"] = dense_head_comparison(x, call_us)
        line["trimmed_head"] = trimmed_head_comparison(x, call_us)
    if world == 1 and not args.no_cpu_baseline and not lowrank:
        x_np = numpy_inputs(x)
        r = oracle_rate(x_np, args.cpu_budget)
        st = single_thread_oracle(args.workload) if not args.no_single_thread else None
        line["cpu_baseline"] = {
            "value": r["value"], "unit": UNIT, "cores": cores(), "kind": "oracle",
            "sample": f"{r['rounds']} whole rounds of the workload ({x['n_calls'] * x['M']} head "
                      f"rows over all {x['V']} vocabulary rows + {x['B']} verified sequences "
                      f"each), {r['seconds']:.1f} s on {cores()} cores",
            "single_thread": ({"value": st["value"], "cores": 1, "rounds": st["rounds"],
                               "seconds": st["seconds"]} if st else None)}
    del x, meas
    torch.cuda.empty_cache()
    if args.workload == "llama8b" and world == 1 and not args.no_workloads:
        # the other configurations, one compact entry each
        line["workloads"] = {}
        for wl in ("gptoss20b", "qwen30b", "specvocab8b"):
            m = measure_round(args, ss, dev, local, world, wl, full=False)
            if not args.no_e2e:
                m["e2e"] = run_e2e(args, m["x"], ss, torch.cuda.Stream(device=dev), world)
            c = compact(m)
            c["config"] = config_dict(wl)
            line["workloads"][wl] = c
            del m
            torch.cuda.empty_cache()
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="llama8b")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--ranks", default=None,
                    help="comma-separated rank per drafted position (one head per position), "
                         "e.g. 768,640,512,512,384,256")
    ap.add_argument("--verify", choices=["logits", "lowrank"], default="logits",
                    help="lowrank: the verifier takes the draft side from the head calls "
                         "(spec_verify_lowrank) instead of draft logits (sampling workloads)")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--clock-seconds", type=float, default=1.5)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-single-thread", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-timeline", action="store_true",
                    help="skip the CUPTI kernel timeline (for runs under ncu, which uses CUPTI "
                         "itself); the line then has no per-kernel figures")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the compact lines of the other configurations (llama8b)")
    ap.add_argument("--no-dense", action="store_true",
                    help="skip the dense V x d head comparison (llama8b)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, world, rank)
        return
    world, rank, local = dist_setup()
    run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
