#!/usr/bin/env python3
"""Benchmark of the drafter-head + verifier hot path on GB300.

One step is one speculative round of the Llama-3.1-8B-shaped workload
(d=4096, r=512, V=128256, M=8 sequences, gamma=6, greedy): gamma low-rank head
calls (each M rows -> M drafted tokens; the drafter backbone between them is
out of scope, so each call gets its own synthetic hidden states) followed by
one greedy verification of the M sequences.  value = drafted tokens/s
(gamma * M per step), whole job over all ranks.

Inputs are resident in HBM; W_up is rotated over gamma copies (one per head
call) so every weight read of the timed region comes from HBM, not L2.
The step is captured in a CUDA graph and replayed.  The dominant kernel's
roofline comes from CUDA events recorded around each library launch on its
own stream (a profiled replay of the same captured step after the timed
region).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle on the host cores, a bounded sample of
the same workload per step.
Multi-GPU: replicas only (the round has no exchange step); one process per
GPU under torchrun, barrier + max-over-ranks timing.
"""
from __future__ import annotations

import argparse
import hashlib
import json
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
        inside = [p for ts, p in rows if t0 <= ts <= t1 + 0.25] or [p for _, p in rows]
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
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4)
                          if p[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside)}


# ------------------------------------------------------------ workload -----
def make_inputs(name: str, seed: int, dev, lowrank: bool = False, head_ranks=None):
    """Seeded synthetic tensors on the device: bf16 weights N(0, 1/fan_in),
    hidden states N(0, 1), Zipf-like target logits (-1.1 ln rank over a random
    permutation + N(0, 0.25)), draft logits = target + N(0, 1).

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
    u_head = [torch.rand(M, generator=g, device=dev) for _ in range(n_calls)]
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
    u_verify = torch.rand(B, gamma + 1, generator=g, device=dev)
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
                w_down=w_down, w_ups=w_ups, u_full=u_full, hidden=hidden, u_head=u_head,
                target=target, lowrank=lowrank, w_downs=w_downs, ranks=head_ranks,
                draft=draft if T > 0 else None, tokens=tokens, u_verify=u_verify)


class Round:
    """Preallocated outputs / workspaces and the step as a sequence of library
    calls on the current stream."""

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

    def head_call(self, j, hidden, u):
        """Head call j of the round (the low-rank head or the SpecVocab head)."""
        x, ss = self.x, self.ss
        T = x["T"]
        if self.specvocab:
            return ss.specvocab_head_forward(hidden, x["w_down"], x["w_ups"][j % len(x["w_ups"])],
                                             x["u_full"], SPECVOCAB_K, T, u if T > 0 else None,
                                             want_topk=False, workspace=self.head_ws,
                                             out=self.head_out[j])
        if self.lowrank:
            return ss.slimspec_head_forward(hidden, x["w_down"], x["w_ups"][0], T, u,
                                            want_stats=True, want_z=True,
                                            workspace=self.head_ws, out=self.head_out[j])
        w_down = x["w_downs"][j] if x.get("w_downs") else x["w_down"]
        return ss.slimspec_head_forward(hidden, w_down, x["w_ups"][j % len(x["w_ups"])], T,
                                        u if T > 0 else None, want_stats=False,
                                        workspace=self.head_ws, out=self.head_out[j])

    def step(self):
        x, ss = self.x, self.ss
        T = x["T"]
        for j in range(x["n_calls"]):
            self.head_call(j, x["hidden"][j], x["u_head"][j])
        if self.lowrank:
            lr = self.lr
            ss.spec_verify_lowrank(x["target"], lr["z"], x["w_ups"][0], lr["logprob"], lr["lse"],
                                   lr["tokens"], T, x["u_verify"], position_major=True,
                                   workspace=self.ver_ws, out=self.ver_out)
            return
        ss.spec_verify(x["target"], x["draft"], x["tokens"], T,
                       x["u_verify"] if T > 0 else None, workspace=self.ver_ws,
                       out=self.ver_out)


def head_stream_bytes(x) -> float:
    """Algorithmic bytes of one up-projection launch (k_head_stream or
    k_head_mma): the W_up stream (V*r*2) and the bf16 z rows it multiplies
    (M*r*2).  Partials are overhead."""
    M, r, V = x["M"], x["r"], x["V"]
    return V * r * 2 + M * r * 2


def verify_rows_read(x, num_accepted) -> int:
    """Rows the accept chain needs (its algorithmic bytes): the target rows of
    positions 0..n_b of each sequence (n_b accepted), and when sampling the
    draft rows of the drafted positions among them.  The row pass reads at
    least these; its roofline is taken against them."""
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
                                      x["u_full"], SPECVOCAB_K, x["T"], x["u_head"][j],
                                      want_topk=True, workspace=rnd.head_ws)
        sizes.append(torch.unique(o["topk_idx"]).numel())
    return float(sum(sizes)) / len(sizes)


def roofline_for(kernel, prof, nbytes, peak, peak_kind, workload):
    n, ms = prof[kernel]
    dur = ms / n / 1000.0
    ach = nbytes / dur / 1e9
    return {"kernel": kernel, "bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s",
            "frac": ach / peak, "traffic": profiled_traffic(kernel, workload),
            "algorithmic_bytes_per_launch": nbytes, "peak_source": peak_kind,
            "us_per_launch": dur * 1e6}


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
            "low_rank_up_projection_us": head_us,
            "speedup_vs_dense": (us / head_us) if head_us else None}


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


# ------------------------------------------------------------ CPU oracle ---
def oracle_round_rate(x_np: dict, budget_s: float, max_steps: int | None = None,
                      steps_exact: int | None = None):
    """Drafted tokens/s of the CPU oracle on bounded samples of the round.

    A sample is one head row (all of W_up's first S rows) plus one verified
    sequence over the same S vocabulary entries; its time is scaled by V/S and
    by the round's gamma*M head rows and B sequences.  S is the largest slice
    whose sample fits the per-step budget.  Returns (rate, steps, S, seconds)."""
    import oracle
    V, M, B, gamma, T = x_np["V"], x_np["M"], x_np["B"], x_np["gamma"], x_np["T"]
    n_rows = x_np["n_calls"] * M

    def sample(S):
        t0 = time.perf_counter()
        if x_np.get("u_full") is not None:   # SpecVocab: router, top-k, gather over S entries
            k_s = max(16, SPECVOCAB_K * S // V)
            oracle.specvocab_head(x_np["hidden"][:1], x_np["w_down"], x_np["w_up"][:S],
                                  x_np["u_full"][:S], k_s, T,
                                  x_np["u_head"][:1] if T > 0 else None)
        else:
            oracle.slimspec_head(x_np["hidden"][:1], x_np["w_down"], x_np["w_up"][:S], "bf16", T,
                                 x_np["u_head"][:1] if T > 0 else None)
        t1 = time.perf_counter()
        tg = x_np["target"][:1, :, :S]
        dr = x_np["draft"][:1, :, :S] if T > 0 else None
        tok = np.minimum(x_np["tokens"][:1], S - 1)
        oracle.verify_batch(tg, dr, tok, x_np["u_verify"][:1] if T > 0 else None, T)
        t2 = time.perf_counter()
        return t1 - t0, t2 - t1

    cal = V if x_np.get("u_full") is None else x_np["u_full"].shape[0]
    th, tv = sample(cal)        # calibration (untimed), on the full row when it is held
    full = (th + tv) * V / cal
    per_step = budget_s if steps_exact is None else budget_s / max(1, steps_exact)
    S = min(cal, V if full <= per_step else max(1024, int(V * per_step / full)))
    steps = steps_exact if steps_exact is not None else max(1, min(max_steps or 10 ** 9,
                                                                  int(budget_s / max(1e-9, full * S / V))))
    tot_h = tot_v = 0.0
    for _ in range(steps):
        a, b = sample(S)
        tot_h += a
        tot_v += b
    round_s = (tot_h / steps * n_rows + tot_v / steps * B) * (V / S)
    return n_rows / round_s, steps, S, tot_h + tot_v


def numpy_inputs(x):
    import torch
    return dict(V=x["V"], M=x["M"], B=x["B"], gamma=x["gamma"], T=x["T"], n_calls=x["n_calls"],
                hidden=x["hidden"][0].float().cpu().numpy(),
                w_down=x["w_down"].float().cpu().numpy(),
                w_up=x["w_ups"][0].float().cpu().numpy(),
                u_head=x["u_head"][0].cpu().numpy(),
                target=x["target"].cpu().numpy(),
                draft=x["draft"].cpu().numpy() if x["draft"] is not None else None,
                tokens=x["tokens"].cpu().numpy(), u_verify=x["u_verify"].cpu().numpy(),
                # SpecVocab's U: the first 32768 rows are as far as a CPU sample reaches
                u_full=(x["u_full"][:32768].float().cpu().numpy()
                        if x["u_full"] is not None else None))


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ----------------------------------------------------------------- arms ---
def run_reference(args, world, rank):
    """CPU oracle arm: rank 0 alone times K steps (after W) of bounded samples."""
    if rank != 0:
        return
    import torch
    # inputs built on the CPU with the same recipe (no GPU needed for this arm)
    dev = torch.device("cpu")
    x = make_inputs(args.workload, 1234, dev)
    x_np = numpy_inputs(x)
    budget = 150.0 / max(1, args.steps + args.warmup)
    oracle_round_rate(x_np, budget * max(1, args.warmup), steps_exact=max(1, args.warmup))
    rate, steps, S, secs = oracle_round_rate(x_np, budget * args.steps, steps_exact=args.steps)
    d, r, V, M, gamma, T = WORKLOADS[args.workload]
    sample = (f"per step: 1 head row + 1 verified sequence over {S} of {V} vocabulary rows, "
              f"scaled to the round ({x['n_calls'] * M} head rows + {x['B']} sequences)")
    # n_gpus is the launch's N; the oracle itself runs on rank 0's host cores only
    line = {"impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * x["n_calls"] * M / rate, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(args.workload),
            "cpu_baseline": {"value": rate, "unit": UNIT, "cores": cores(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


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
            "low_rank_up_projection_us": head_us,
            "note": "the low-rank head scores all V rows; the trimmed head never drafts the "
                    f"{V - kept} dropped ids"}


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
    x = make_inputs(args.workload, 1234 + rank, dev, lowrank=lowrank, head_ranks=ranks)
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

    sampler = ClockSampler(local) if not args.no_clocks else None
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
    wall1 = time.time()
    torch.cuda.synchronize()
    barrier(world)
    if sampler:
        sampler.stop()
    sec_local = e0.elapsed_time(e1) / 1000.0
    units, secs = aggregate(units_per_step * args.steps, sec_local, world)
    value = units / secs
    assert ss.ss_get_device_error() == ss.SS_OK
    step_dist = step_time_distribution(graph, stream, min(args.steps, 500))

    # per-kernel device time: the step captured again with the library's
    # event pairs around every launch, replayed and read after each replay
    ss.profile_start()
    pgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(pgraph, stream=stream, capture_error_mode="thread_local"):
        rnd.step()
    ss.profile_stop()
    n_prof = min(50, max(5, args.steps))
    prof = {}
    for _ in range(n_prof):
        with torch.cuda.stream(stream):
            pgraph.replay()
        stream.synchronize()
        for name, (n, ms) in ss.profile_read(keep=True).items():
            a = prof.setdefault(name, [0, 0.0])
            a[0] += n
            a[1] += ms
    ss.profile_read(keep=False)
    prof = {k: tuple(v) for k, v in prof.items()}

    # end to end through the public API with host buffers
    e2e = run_e2e(args, x, ss, stream, world) if not args.no_e2e else None

    if rank != 0:
        return
    kern = {}
    total_ms = sum(ms for _, ms in prof.values())
    for name, (n, ms) in sorted(prof.items(), key=lambda kv: -kv[1][1]):
        kern[name] = {"launches_per_step": n / n_prof, "us_per_launch": 1000.0 * ms / n,
                      "share": ms / total_ms}
    # the dominant kernel (largest share of the step among the kernels with
    # algorithmic bytes), the head's up-projection, and the verifier's row pass
    peak, peak_kind = measured_peaks()
    kb = kernel_bytes(x, union_rows, ver_rows)
    if "k_verify_rows" in prof:
        # the row pass may be split in two launches (position 0, then the
        # positions of the sequences that kept it): the bytes are per step
        kb["k_verify_rows"] /= prof["k_verify_rows"][0] / n_prof
    cands = [k for k in prof if k in kb]
    roof = head_roof = ver_roof = None
    if cands:
        dom = max(cands, key=lambda k: prof[k][1])
        roof = roofline_for(dom, prof, kb[dom], peak, peak_kind, args.workload)
    head_kernel = next((k for k in ("k_head_mma", "k_head_stream") if k in prof), None)
    if head_kernel:
        head_roof = roofline_for(head_kernel, prof, kb[head_kernel], peak, peak_kind, args.workload)
        if head_kernel == "k_head_mma":
            flops = 2.0 * x["M"] * x["V"] * x["r"]
            tpeak = measured_tensor_peak()
            dur = head_roof["us_per_launch"] / 1e6
            head_roof["tensor"] = {"achieved": flops / dur / 1e12, "peak": tpeak,
                                   "unit": "TFLOP/s", "frac": flops / dur / 1e12 / tpeak,
                                   "algorithmic_flops_per_launch": flops}
            if roof and roof["kernel"] == head_kernel:
                roof["tensor"] = head_roof["tensor"]
    if "k_verify_rows" in prof:
        ver_roof = roofline_for("k_verify_rows", prof, kb["k_verify_rows"], peak, peak_kind,
                                args.workload)
        ver_roof["launches_per_step"] = prof["k_verify_rows"][0] / n_prof
        ver_roof["rows_needed"] = ver_rows
        ver_roof["rows_total"] = x["B"] * (x["gamma"] + 1) + (
            x["B"] * x["gamma"] if x["T"] > 0 and not x.get("lowrank", False) else 0)
    ver_ms = sum(ms for name, (n, ms) in prof.items() if name.startswith("k_verify")) / n_prof
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs * 1000.0 / args.steps,
            "ms_per_step_dist": step_dist,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic: seeded N(0,1/fan_in) bf16 weights, N(0,1) hidden states, "
                    "Zipf-like target logits",
            "config": dict(config_dict(args.workload), **(
                {"verify": "draft side from the head calls (z, log q, lse; spec_verify_lowrank), "
                           "one W_up for all calls"} if lowrank else {}),
                **({"ranks_per_position": ranks} if ranks else {})), "roofline": roof,
            "head_roofline": head_roof, "verify_roofline": ver_roof,
            "specvocab_union_rows": union_rows if x["u_full"] is not None else None,
            "gpu_launches": int(launches_per_step * args.steps),
            "verify_steps_per_s": (1000.0 / ver_ms) if ver_ms > 0 else None,
            "kernels": kern}
    if sampler:
        line["clocks"] = sampler.summary(wall0, wall1)
    if e2e:
        line["e2e"] = e2e
    if args.workload == "llama8b" and not args.no_dense:
        # the Llama-shaped configuration also names the dense 128256 x 4096 head
        line["dense_head"] = dense_head_comparison(
            x, head_roof["us_per_launch"] if head_roof else None)
        line["trimmed_head"] = trimmed_head_comparison(
            x, head_roof["us_per_launch"] if head_roof else None)
    if world == 1 and not args.no_cpu_baseline:
        x_np = numpy_inputs(x)
        rate, steps, S, secs_cpu = oracle_round_rate(x_np, args.cpu_budget)
        line["cpu_baseline"] = {
            "value": rate, "unit": UNIT, "cores": cores(), "kind": "oracle",
            "sample": f"{steps} samples of 1 head row + 1 verified sequence over {S} of "
                      f"{x['V']} vocabulary rows ({secs_cpu:.1f} s of CPU work), scaled to the "
                      f"round ({units_per_step} head rows + {x['B']} sequences)"}
    print(json.dumps(line), flush=True)


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


def run_e2e(args, x, ss, stream, world):
    """Same round through the Python API with pinned host inputs copied in and
    the tokens copied out inside the timed region, every step.

    The drafting calls' inputs (hidden rows, uniforms) are packed in one host
    buffer each and copied first on the launching stream; the verifier's
    inputs (target and draft rows, tokens, uniforms) are then copied on a
    second stream that overlaps the drafting calls, and the verifier waits
    for it.  In this synthetic round both sets of inputs are
    independent host arrays, so nothing orders the second copy after the
    drafting calls."""
    import torch
    dev = x["w_down"].device
    T, M, n_calls, B, gamma = x["T"], x["M"], x["n_calls"], x["B"], x["gamma"]
    lowrank = x.get("lowrank", False)
    h_host = torch.stack([h.cpu() for h in x["hidden"]]).pin_memory()
    u_host = torch.stack([u.cpu() for u in x["u_head"]]).pin_memory()
    h_dev = torch.empty_like(h_host, device=dev)
    u_dev = torch.empty_like(u_host, device=dev)
    # the verifier's host inputs: target rows always; draft rows and tokens
    # unless the draft side comes from the drafting calls
    v_host = {"target": x["target"].cpu().pin_memory()}
    if T > 0:
        v_host["u_verify"] = x["u_verify"].cpu().pin_memory()
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
    copy_stream = torch.cuda.Stream(device=dev)
    started = torch.cuda.Event()
    copied = torch.cuda.Event()

    def step():
        # the drafting inputs first: a copy queued behind the verifier's rows
        # on the same copy engine would hold the drafting calls back
        h_dev.copy_(h_host, non_blocking=True)
        if T > 0:
            u_dev.copy_(u_host, non_blocking=True)
        # the verifier's copy starts after them; the previous step's verifier,
        # earlier on the launching stream, has finished with its buffers
        started.record(stream)
        copy_stream.wait_event(started)
        with torch.cuda.stream(copy_stream):
            for k in v_host:
                v_dev[k].copy_(v_host[k], non_blocking=True)
            copied.record(copy_stream)
        for j in range(n_calls):
            rnd.head_call(j, h_dev[j], u_dev[j])
        stream.wait_event(copied)
        if lowrank:
            lr = rnd.lr
            ss.spec_verify_lowrank(v_dev["target"], lr["z"], x["w_ups"][0], lr["logprob"],
                                   lr["lse"], lr["tokens"], T, v_dev["u_verify"],
                                   position_major=True, workspace=rnd.ver_ws, out=ver_out)
        else:
            ss.spec_verify(v_dev["target"], v_dev.get("draft"), v_dev["tokens"], T,
                           v_dev.get("u_verify"), workspace=rnd.ver_ws, out=ver_out)
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
    copy_stream.synchronize()
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
    if T > 0:
        h2d += u_host.numel() * u_host.element_size()
    return {"value": units / secs, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(out_host.numel() * 4), "steps": n_steps,
            "issue": "the step's copies and calls captured once in a CUDA graph, replayed per step",
            "eager_value": eager_units / eager_secs,
            "verifier_inputs_copy": "second stream, overlapping the drafting calls"}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="llama8b")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--ranks", default=None,
                    help="comma-separated rank per drafted position (one head per position), "
                         "e.g. 768,640,512,512,384,256")
    ap.add_argument("--verify", choices=["logits", "lowrank"], default="logits",
                    help="lowrank: the verifier takes the draft side from the head calls "
                         "(spec_verify_lowrank) instead of draft logits (sampling workloads)")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
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
