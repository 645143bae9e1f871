#!/usr/bin/env python
"""Throughput of the Dust estimator engine on B300: perturbed token-evaluations/s.

One step is one call of an estimator entry point over one batch: every step
of the hot path (noise, perturbed loss, centring/reward, error estimate, outer
product) runs inside it.  The metric is draws x tokens per second.

Default workload: the LM-head estimator at the pages' batch shape -- 8
sequences x 2048 tokens, d = 512, vocabulary 4096, K = 64 draws, sigma = 0.05
(linlog.top article, experimental setup; Dust translation, hn.213312.xyz,
§3.1).  Inputs are synthetic: Zipf(1.1) targets stand in for FineWeb token
frequencies; weights are random N(0, 1/fan_in).  The cached logits (256 MB)
are larger than the 126 MB L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl dust|reference]
                  [--workload head_batch|head_batch_antithetic|head_batch_chunked|head_tiny|
                              head_scale|interior|
                              interior_scale|embed_scale|head_sweep|optim_adam|attn_value|
                              attn_qk]

Under torchrun (N > 1) every rank estimates its own batch (global token
offset rank * T, so the noise differs per rank), and each step ends with the
step's one exchange, the sum of the ranks' weight gradients (an NCCL
all-reduce of G_W, inside the timed step); rank 0 prints the aggregate over
the slowest rank's time.

--impl reference times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload (the pages give no implementation to run).
"""
import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("perturbed token-evals/sec (draws×tokens/s) on 1 B300; "
          "% of HBM/tensor roofline")
UNIT = "token-evals/s"
N_SM = 148
SM_MAX_MHZ = 2032.0
# Algorithmic operation budget of one head element-draw (one noise sample, one
# perturbed probability term, two accumulator updates), counted in the design
# notes: Philox 9 + uniform 2 + Box-Muller 3 + CE 2 + accumulators 2 + share
# of the per-draw reduction 2.
HEAD_OPS_PER_ELEMENT_DRAW = 20
# antithetic pair: one noise value (Philox 9, uniform 2, Box-Muller 3), two loss
# terms (4), one accumulator, reduction share 2
HEAD_OPS_PER_ELEMENT_PAIR = 21


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
                "sm_max_mhz": SM_MAX_MHZ}, "fallback"


class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def rank_token0(rank, tokens_per_rank):
    """Global index of a rank's first token: every rank estimates its own
    batch, and the noise (keyed by global token) differs between ranks."""
    return rank * tokens_per_rank


def max_over_ranks(value, dist=None):
    """The slowest rank's value (the job's time); the value itself on one rank."""
    import torch
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------- workloads ----
def make_workload(name, device, rank):
    import torch

    import workloads as W
    bf = torch.bfloat16
    dev = lambda a, dt=None: (torch.from_numpy(np.ascontiguousarray(a)).to(device)
                              if dt is None else torch.from_numpy(np.ascontiguousarray(a)).to(device).to(dt))
    if name.startswith("head"):
        p = W.HEAD_PARAMS[name]
        wl = W.head_workload(p["T"], p["d"], p["V"], p["seq_len"], p["x_bf16"], p["zipf"],
                             device=str(device))
        T = p["T"]
        return {
            "kind": "head", "name": name, "T": T, "V": p["V"], "d": p["d"], "K": p["K"],
            "sigma": p["sigma"], "seq_len": p["seq_len"], "token0": rank_token0(rank, T),
            "baseline": p.get("baseline", 0), "vchunk": p.get("chunk", 0),
            "host": {"logits": wl["z"], "targets": wl["targets"],
                     "x": W.bf16_round(wl["x"]) if p["x_bf16"] else wl["x"]},
            "x_bf16": p["x_bf16"],
            "dev": {"logits": dev(wl["z"]), "targets": dev(wl["targets"]),
                    "x": dev(wl["x"], bf) if p["x_bf16"] else dev(wl["x"])},
        }
    if name.startswith("interior"):
        p = W.INTERIOR_PARAMS[name]
        wl = W.interior_workload(p["T"], p["d_in"], p["C"], p["d_model"], p["V"], p["seq_len"],
                                 device=str(device))
        return {
            "kind": "interior", "name": name, "T": p["T"], "K": p["K"], "sigma": p["sigma"],
            "gamma": p["gamma"], "seq_len": p["seq_len"], "lam": wl["lam"], "C": p["C"],
            "d_in": p["d_in"], "d_model": p["d_model"], "V": p["V"],
            "token0": rank_token0(rank, p["T"]),
            "host": {k: wl[k] for k in ("x", "y1", "W2", "W_head", "z_clean", "targets")},
            "dev": {"x": dev(wl["x"], bf), "y1": dev(wl["y1"]), "W2": dev(wl["W2"], bf),
                    "W_head": dev(wl["W_head"], bf), "z_clean": dev(wl["z_clean"]),
                    "targets": dev(wl["targets"])},
        }
    if name == "embed_scale":
        wl = W.embed_workload()
        # g (101 MB) is smaller than L2: the steps rotate over three copies of
        # the inputs, so a step's inputs were last read two steps (200 MB) ago
        return {"kind": "embed", "name": name, "T": wl["T"], "d": wl["d"], "V": wl["V"], "K": 1,
                "host": {"g": wl["g"], "ids": wl["ids"]}, "rotate": 3,
                "dev": {"g": dev(wl["g"]), "ids": dev(wl["ids"])}}
    raise SystemExit("unknown workload " + name)


def make_step(wl, dust):
    """Returns (step(), evals per step, launches per step, workspace, G_W) with
    outputs and workspace allocated once."""
    import torch
    d = wl["dev"]
    if wl["kind"] == "head":
        T, V, dd, K = wl["T"], wl["V"], wl["d"], wl["K"]
        g = torch.empty((T, V), dtype=torch.float32, device=d["logits"].device)
        G = torch.empty((V, dd), dtype=torch.float32, device=g.device)
        ws = dust._workspace(dust.head_workspace_bytes(T, V, dd, K), g.device)

        if wl["vchunk"]:
            ws = dust._workspace(dust.lib().dust_head_chunked_workspace(T, V, dd, K, wl["vchunk"]),
                                 g.device)

            def step():
                dust.head_estimate_chunked(d["logits"], d["targets"], d["x"], wl["sigma"], K, 1234,
                                           wl["vchunk"], token0=wl["token0"], out=(g, G), ws=ws)
            # lse, one draw kernel per chunk, the outer product
            return step, K * T, 2 + V // wl["vchunk"], ws, G

        def step():
            dust.head_estimate(d["logits"], d["targets"], d["x"], wl["sigma"], K, 1234, 0, 0,
                               wl["token0"], out=(g, G), ws=ws, baseline=wl["baseline"])
        launches = 2 + (0 if wl["x_bf16"] else 1)
        # antithetic pairs: two perturbed evaluations per noise draw
        return step, K * T * (2 if wl["baseline"] == 2 else 1), launches, ws, G
    if wl["kind"] == "interior":
        T, K = wl["T"], wl["K"]
        g = torch.empty((T, wl["C"]), dtype=torch.float32, device=d["x"].device)
        G = torch.empty((wl["C"], wl["d_in"]), dtype=torch.float32, device=g.device)
        ws = dust._workspace(dust.linear_workspace_bytes(T, wl["d_in"], wl["C"], wl["d_model"],
                                                          wl["V"], K), g.device)

        def step():
            dust.linear_estimate(d["x"], d["y1"], d["W2"], wl["lam"], d["W_head"], d["z_clean"],
                                 d["targets"], wl["seq_len"], wl["sigma"], wl["gamma"], K, 1234,
                                 1, 0, wl["token0"], out=(g, G), ws=ws)
        # draws per chunk as the library plans them: >= 8 tiles per SM, a
        # whole number of waves over 148 SMs where possible
        ntb = -(-T // 128)
        nd = -(-1184 // ntb)
        for c in range(nd, min(64, 4 * nd) + 1):
            if (c * ntb) % 148 == 0:
                nd = c
                break
        nd = max(1, min(nd, 64, K))
        chunks = -(-K // nd)
        fused = wl["C"] % 64 == 0 and wl["d_model"] <= 512
        # GEMM 1 (+ EMA in its epilogue for whole token blocks per sequence), GEMM 2
        per_chunk = (2 if wl["seq_len"] % 128 == 0 else 3) if fused else 4
        # softmax (+ clean GELU when fused), per chunk, mean + scan + g, outer product
        return step, K * T, (2 if fused else 1) + chunks * per_chunk + 3 + 1, ws, G
    if wl["kind"] == "embed":
        T, dd, V = wl["T"], wl["d"], wl["V"]
        G = torch.empty((V, dd), dtype=torch.float32, device=d["g"].device)
        perm = torch.empty(T, dtype=torch.int32, device=G.device)
        ws = dust._workspace(dust.embed_workspace_bytes(T, dd, V), G.device)
        sets = [d] + [{k: v.clone() for k, v in d.items()} for _ in range(wl.get("rotate", 1) - 1)]
        cur = [0]

        def step():
            s_ = sets[cur[0]]
            cur[0] = (cur[0] + 1) % len(sets)
            dust.embed_scatter(s_["g"], s_["ids"], V, out=(G, perm), ws=ws)
        return step, T, 4, ws, G
    raise SystemExit("bad workload")


def issue_probes(dust):
    """Measured issue rates (T operations/s) of the library's probe kernel:
    Philox's multiply/xor step, ex2 on the XU pipe, and fp32 fma."""
    out = {}
    for kind, name, iters in ((0, "philox_mul_xor", 10000), (1, "ex2", 4000), (2, "ffma", 40000),
                              (5, "ffma2_ops", 40000)):
        dust.issue_probe(kind, 16)  # warm-up
        rate, _ = dust.issue_probe(kind, iters)
        out[name] = rate / 1e12
    out["unit"] = "Tops/s"
    return out


def interior_kernel_split(times_ms, steps):
    """The interior call's timed launches per step: GEMM 1 and GEMM 2 (+ CE)
    alternating once per chunk of draws, then the credit and g pass.  Returns
    (GEMM 1 ms, GEMM 2 ms, credit + g ms) per step."""
    per = len(times_ms) // max(steps, 1)
    if per < 3 or per % 2 == 0:
        return None, None, None
    g1 = g2 = gp = 0.0
    for st in range(steps):
        t = times_ms[st * per:(st + 1) * per]
        g1 += sum(t[0:per - 1:2])
        g2 += sum(t[1:per - 1:2])
        gp += t[per - 1]
    return g1 / steps, g2 / steps, gp / steps


def roofline(wl, kernel_ms, traffic, probes=None, split=None):
    peaks, which = _peaks()
    if wl["kind"] == "head":
        per = HEAD_OPS_PER_ELEMENT_PAIR if wl.get("baseline") == 2 else HEAD_OPS_PER_ELEMENT_DRAW
        width = wl.get("vchunk") or wl["V"]  # elements perturbed per draw
        ops = per * wl["T"] * width * wl["K"]
        peak = N_SM * 128 * peaks.get("sm_max_mhz", SM_MAX_MHZ) * 1e6 / 1e12
        ach = ops / (kernel_ms * 1e-3) / 1e12
        return {"bound": "alu", "achieved": ach, "peak": peak, "unit": "Tops/s",
                "frac": ach / peak, "traffic": traffic,
                "kernel": ("head_draws_kernel<antithetic>" if wl.get("baseline") == 2 else
                           "head_draws_kernel<vocabulary chunks>" if wl.get("vchunk") else
                           "head_pair_kernel"),
                "kernel_ms": kernel_ms, "peak_source": "148 SMs x 128 lanes x %.0f MHz (%s clocks)"
                % (peaks.get("sm_max_mhz", SM_MAX_MHZ), which),
                "issue_probe": probes}
    if wl["kind"] == "interior":
        # Algorithmic flops: one product per multiply-add of the method's own
        # contractions (the split-bf16 kernels execute twice that).
        #   GEMM 2 (+ CE): K draws x T rows x d_model x V
        #   GEMM 1:        K draws x T rows x C x d_model
        g1_ms, g2_ms, gp_ms = split if split else (None, kernel_ms, None)
        peak = peaks["bf16_tflops_sustained"]
        f2 = 2.0 * wl["K"] * wl["T"] * wl["d_model"] * wl["V"]
        f1 = 2.0 * wl["K"] * wl["T"] * wl["C"] * wl["d_model"]
        ach = f2 / (g2_ms * 1e-3) / 1e12
        out = {"bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
               "frac": ach / peak, "traffic": traffic,
               "kernel": "gemm_bf16_kernel<CE> (GEMM 2 + cross-entropy)",
               "kernel_ms": g2_ms, "flops": "algorithmic (split-bf16 executes 2x)",
               "peak_source": "bf16_tflops_sustained (%s)" % which}
        if g1_ms:
            a1 = f1 / (g1_ms * 1e-3) / 1e12
            out["gemm1"] = {"kernel": "reforward1_kernel (GEMM 1 + EMA)", "kernel_ms": g1_ms,
                            "achieved": a1, "frac": a1 / peak}
            out["credit_and_g_ms"] = gp_ms
        return out
    if wl["kind"] == "embed":
        # what the whole call must move: every g row read once, the ids read
        # and the permutation written, every G_E row written once; over the
        # device time of the whole call (its memset and four kernels)
        nbytes = wl["T"] * wl["d"] * 4 + wl["T"] * 4 * 2 + wl["V"] * wl["d"] * 4
        peak = peaks["hbm_gbs"]
        ach = nbytes / (kernel_ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
                "traffic": traffic, "kernel": "the whole embedding call (memset, sort, rows)",
                "kernel_ms": kernel_ms, "bytes_per_call": nbytes,
                "peak_source": "hbm_gbs (%s)" % which}
    return None


def load_traffic(wl):
    """Per-launch DRAM bytes of the dominant kernel from a committed ncu
    capture, if the capture's kernel source still matches."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(wl["name"])
    except (OSError, ValueError):
        return None
    if not rec:
        return None
    h = hashlib.sha256()
    for src in rec.get("sources", []):
        try:
            h.update(open(os.path.join(ROOT, src), "rb").read())
        except OSError:
            return None
    if h.hexdigest() != rec.get("sha256"):
        return None
    return rec.get("bytes_per_launch")


# ------------------------------------------------------------ CPU oracle ----
def oracle_sample(wl, budget_s=12.0):
    """The fp64 oracle on a bounded slice of the workload: (evals/s, sample text)."""
    import oracle
    h = wl["host"]
    if wl["kind"] == "head":
        K = wl["K"]
        anti = wl.get("baseline") == 2
        fn = oracle.head_estimate_antithetic if anti else oracle.head_estimate

        def run(n):
            t0 = time.perf_counter()
            if wl.get("vchunk"):
                oracle.head_estimate_chunked(h["logits"][:n], h["targets"][:n], h["x"][:n],
                                             wl["sigma"], K, 1234, 0, wl["vchunk"])
            else:
                fn(h["logits"][:n], h["targets"][:n], h["x"][:n], wl["sigma"], K, 1234, 0, 0, 0)
            return time.perf_counter() - t0
        n = 8
        dt = run(n)
        n = int(min(wl["T"], max(8, n * budget_s / max(dt, 1e-3))))
        dt = run(n)
        return K * n * (2 if anti else 1) / dt, "%d of %d tokens, all %d draws%s, full " \
            "vocabulary %d" % (n, wl["T"], K, " (antithetic pairs)" if anti else "", wl["V"])
    if wl["kind"] == "interior":
        L = wl["seq_len"]

        def run(k):
            t0 = time.perf_counter()
            oracle.linear_estimate(h["x"][:L], h["y1"][:L], h["W2"], wl["lam"], h["W_head"],
                                   h["z_clean"][:L], h["targets"][:L], L, wl["sigma"],
                                   wl["gamma"], k, 1234, 1, 0, 0)
            return time.perf_counter() - t0
        k = 2
        dt = run(k)
        k = int(min(wl["K"], max(2, k * budget_s / max(dt, 1e-3))))
        dt = run(k)
        return k * L / dt, "sequence 0 (%d tokens), %d of %d draws" % (L, k, wl["K"])
    if wl["kind"] == "embed":
        t0 = time.perf_counter()
        oracle.embed_scatter(h["g"], h["ids"], wl["V"])
        dt = time.perf_counter() - t0
        return wl["T"] / dt, "whole workload (%d tokens)" % wl["T"]
    return None, ""


L2_BYTES = 126 << 20
FLUSH_BYTES = 256 << 20


def input_bytes(wl):
    return sum(np.asarray(v).nbytes for v in wl["host"].values())


def l2_mode(wl):
    """How a step's inputs are kept out of L2: "large" (the inputs are larger
    than L2), "rotate" (the steps rotate over copies of the inputs) or "flush"
    (a 256 MB write before every step, outside the step's events)."""
    if wl.get("rotate", 1) > 1:
        return "rotate"
    return "large" if input_bytes(wl) > L2_BYTES else "flush"


def l2_label(wl):
    mode = l2_mode(wl)
    if mode == "rotate":
        n = wl["rotate"]
        return "%d input sets of %.0f MB rotated (%.0f MB > L2)" % (
            n, input_bytes(wl) / 1e6, n * input_bytes(wl) / 1e6)
    if mode == "flush":
        return "L2 flushed before every step (a 256 MB write outside the step's events)"
    return "inputs larger than L2 (no flush)"


class StepTimer:
    """Device time of n calls of fn on a stream.  Without a flush, one pair of
    events brackets all the calls; with one, a 256 MB write precedes every
    call and a pair of events brackets each call alone (their sum)."""

    def __init__(self, stream, flush):
        import torch
        self.stream = stream
        self.scrub = (torch.empty(FLUSH_BYTES // 4, dtype=torch.int32, device=stream.device)
                      if flush else None)

    def flush(self):
        if self.scrub is not None:
            self.scrub.fill_(1)

    def time(self, n, fn):
        import torch
        ev = lambda: torch.cuda.Event(enable_timing=True)
        if self.scrub is None:
            e0, e1 = ev(), ev()
            e0.record(self.stream)
            for _ in range(n):
                fn()
            e1.record(self.stream)
            e1.synchronize()
            return e0.elapsed_time(e1)
        pairs = []
        for _ in range(n):
            self.flush()
            a, b = ev(), ev()
            a.record(self.stream)
            fn()
            b.record(self.stream)
            pairs.append((a, b))
        pairs[-1][1].synchronize()
        return sum(a.elapsed_time(b) for a, b in pairs)


def config_of(wl, n_gpus):
    c = {"workload": wl["name"], "tokens": wl["T"], "draws": wl["K"],
         "l2": l2_label(wl), "parallelism": "dp%d" % n_gpus}
    if n_gpus > 1:
        c["tokens_per_rank"] = wl["T"]
        c["exchange"] = "G_W summed over ranks (all-reduce) every step"
    for k in ("V", "d", "C", "d_in", "d_model", "seq_len", "sigma", "gamma"):
        if k in wl:
            c[k] = wl[k]
    if wl.get("baseline") == 2:
        c["baseline"] = "antithetic pairs: draws counts noise draws, 2 evaluations each"
    if wl.get("vchunk"):
        c["vocab_chunk"] = wl["vchunk"]
    return c


OPTIM_PARAMS = 38_000_000  # the pages' 8-layer, 512-wide GPT has about 38M parameters
OPTIM_BYTES_PER_PARAM = 4 * 7 + 2  # W, m, v read and written, G read (fp32); bf16 W out


def run_optim(args):
    """The optimiser step that consumes the estimate (Adam with decoupled
    weight decay, writing the bf16 copy of W), over all parameters of the
    pages' 38M-parameter GPT at once, inputs resident: parameter updates/s
    and the fraction of the HBM roofline at 30 bytes per parameter."""
    import torch

    import activation_perturbation_es_noise_b300 as dust
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    n = OPTIM_PARAMS
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    Wt = torch.randn(n, device=dev, generator=gen)
    G = torch.randn(n, device=dev, generator=gen)
    m = torch.zeros(n, device=dev)
    v = torch.zeros(n, device=dev)
    Wb = torch.empty(n, dtype=torch.bfloat16, device=dev)
    t = [0]

    def step():
        t[0] += 1
        dust.adam_step(Wt, G, m, v, t[0], 1e-3, weight_decay=0.01, W_bf16=Wb)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clocks:
        for _ in range(max(3, args.warmup)):  # clocks back up after the sampler's start
            step()
        torch.cuda.synchronize()
        e0.record()
        for _ in range(args.steps):
            step()
        e1.record()
        e1.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    peaks, which = _peaks()
    ach = OPTIM_BYTES_PER_PARAM * n / (ms * 1e-3) / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        k = 200_000
        a = [np.random.default_rng(1).standard_normal(k) for _ in range(2)]
        t0 = time.perf_counter()
        oracle.adam_step(a[0], a[1], np.zeros(k), np.zeros(k), 1, 1e-3, 0.9, 0.999, 1e-8, 0.01)
        cpu = {"value": k / (time.perf_counter() - t0), "unit": "params/s", "cores": 1,
               "kind": "oracle", "sample": "%d of %d parameters, one step" % (k, n)}
    print(json.dumps({
        "metric": "optimiser parameter updates/sec (Adam step) on 1 B300; % of HBM roofline",
        "value": n / (ms * 1e-3), "unit": "params/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "optim_adam", "params": n, "l2": "inputs larger than L2 (no flush)"},
        "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": ach / peaks["hbm_gbs"], "traffic": load_traffic({"name": "optim_adam"}),
                     "kernel": "optim_kernel<Adam>", "kernel_ms": ms,
                     "peak_source": "hbm_gbs (%s)" % which},
        "cpu_baseline": cpu, "e2e": None, "gpu_launches": args.steps,
        "clocks": clocks.summary()}), flush=True)
    return 0


ATTN = dict(nseq=8, H=8, L=2048, d_in=512, K=64, sigma=0.02, gamma=0.99)


def run_attn_value(args):
    """The value projection inside attention (8 x 2048 tokens, 8 heads of 64,
    d_in 512, K = 64, gamma 0.99), inputs resident: token-evals/s, and the
    re-forward kernel against the sustained bf16 tensor peak on the method's
    own flops: per (sequence, head, draw), the causal product
    sum_{t <= s} P[s, t] a_t, 64 multiply-adds for each of the L (L + 1) / 2
    (query, key) pairs.  The kernel executes three split-bf16 passes over whole
    128-key tiles up to the diagonal (the line's `executed_tflop`)."""
    import torch

    import activation_perturbation_es_noise_b300 as dust
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    c = ATTN
    nseq, H, L, K = c["nseq"], c["H"], c["L"], c["K"]
    T = nseq * L
    gen = torch.Generator(device=dev)
    gen.manual_seed(21)
    s = torch.randn((nseq, H, L, L), generator=gen, device=dev) * 2.0
    s = s.masked_fill(torch.triu(torch.ones(L, L, dtype=torch.bool, device=dev), 1), -1e30)
    P = torch.softmax(s, dim=-1).contiguous()
    del s
    E = torch.randn((T, H * 64), generator=gen, device=dev) * 0.1
    x = torch.randn((T, c["d_in"]), generator=gen, device=dev).to(torch.bfloat16)
    g = torch.empty((T, H * 64), dtype=torch.float32, device=dev)
    G = torch.empty((H * 64, c["d_in"]), dtype=torch.float32, device=dev)
    ws = dust._workspace(dust.lib().dust_attn_value_workspace(T, L, H, 64, c["d_in"], K), dev)

    def step():
        dust.attn_value_estimate(P, E, x, L, c["sigma"], c["gamma"], K, 1234, out=(g, G), ws=ws)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clocks:
        for _ in range(max(3, args.warmup)):  # clocks back up after the sampler's start
            step()
        torch.cuda.synchronize()
        e0.record()
        for _ in range(args.steps):
            step()
        e1.record()
        e1.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    timer = dust.KernelTimer(capacity=args.steps * (K // 4 + 1))
    with timer:
        torch.cuda._sleep(1_000_000 * args.steps)
        for _ in range(args.steps):
            step()
    torch.cuda.synchronize()
    kernel_ms = timer.total_ms() / args.steps
    # covered key slices per (sequence, head): sum over query tiles of 128 x 128 (qb + 1)
    nt = L // 128
    pairs = 128 * 128 * nt * (nt + 1) // 2
    executed = 3 * 2.0 * pairs * 64 * 4 * (K // 4) * nseq * H
    flops = 2.0 * 64 * (L * (L + 1) // 2) * K * nseq * H
    peaks, which = _peaks()
    ach = flops / (kernel_ms * 1e-3) / 1e12
    print(json.dumps({
        "metric": METRIC, "value": K * T / (ms * 1e-3), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32+bf16x3", "data": "synthetic",
        "config": {"workload": "attn_value", "tokens": T, "draws": K, "heads": H, "dv": 64,
                   "d_in": c["d_in"], "seq_len": L, "sigma": c["sigma"], "gamma": c["gamma"],
                   "l2": "inputs larger than L2 (no flush)"},
        "roofline": {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops_sustained"],
                     "unit": "TFLOP/s", "frac": ach / peaks["bf16_tflops_sustained"],
                     "traffic": load_traffic({"name": "attn_value"}), "kernel": "attn_v_kernel",
                     "kernel_ms": kernel_ms, "flops": "algorithmic",
                     "algorithmic_tflop": flops / 1e12, "executed_tflop": executed / 1e12,
                     "peak_source": "bf16_tflops_sustained (%s)" % which},
        "cpu_baseline": None, "e2e": None, "gpu_launches": args.steps * (2 * (K // 4) + 6),
        "clocks": clocks.summary()}), flush=True)
    return 0


def run_attn_qk(args):
    """The query projection inside attention (which 0; 8 x 2048 tokens, 8
    heads of 64, d_in 512, K = 64, gamma 0.99), inputs resident: token-evals/s,
    and the tensor-core kernel against the sustained bf16 peak on the method's
    own flops: per (sequence, head, draw) and causal (query, key) pair, two
    64-long dot products (the score shift and the weighted value).  The kernel
    executes each over whole 64-key slices up to the diagonal as three
    split-bf16 passes (the line's `executed_tflop`)."""
    import torch

    import activation_perturbation_es_noise_b300 as dust
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    c = ATTN
    nseq, H, L, K = c["nseq"], c["H"], c["L"], c["K"]
    T, C = nseq * L, H * 64
    gen = torch.Generator(device=dev)
    gen.manual_seed(22)
    Q, Kk, V = (torch.randn((T, C), generator=gen, device=dev) for _ in range(3))
    q4, k4, v4 = (t.view(nseq, L, H, 64).transpose(1, 2) for t in (Q, Kk, V))
    s = (q4 @ k4.transpose(-1, -2)) / 8.0
    s = s.masked_fill(torch.triu(torch.ones(L, L, dtype=torch.bool, device=dev), 1), -1e30)
    P = torch.softmax(s, dim=-1).contiguous()
    del s
    O = (P @ v4).transpose(1, 2).reshape(T, C).contiguous()
    E = torch.randn((T, C), generator=gen, device=dev) * 0.1
    x = torch.randn((T, c["d_in"]), generator=gen, device=dev).to(torch.bfloat16)
    g = torch.empty((T, C), dtype=torch.float32, device=dev)
    G = torch.empty((C, c["d_in"]), dtype=torch.float32, device=dev)
    ws = dust._workspace(dust.lib().dust_attn_qk_workspace(T, L, H, 64, c["d_in"], K), dev)

    def step():
        dust.attn_qk_estimate(0, Q, Kk, V, O, P, E, x, L, c["sigma"], c["gamma"], K, 1234,
                              out=(g, G), ws=ws)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clocks:
        for _ in range(max(3, args.warmup)):  # clocks back up after the sampler's start
            step()
        torch.cuda.synchronize()
        e0.record()
        for _ in range(args.steps):
            step()
        e1.record()
        e1.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    timer = dust.KernelTimer(capacity=args.steps + 1)
    with timer:
        torch.cuda._sleep(1_000_000 * args.steps)
        for _ in range(args.steps):
            step()
    torch.cuda.synchronize()
    kernel_ms = timer.total_ms() / args.steps
    nt = L // 128
    slices = 2 * nt * (nt + 1) // 2  # 64-key slices per (sequence, head, draw)
    executed = 3 * 2 * (2.0 * 128 * 64 * 64) * slices * nseq * H * K
    flops = 2 * 2.0 * 64 * (L * (L + 1) // 2) * nseq * H * K
    peaks, which = _peaks()
    peak = peaks["bf16_tflops_sustained"]
    ach = flops / (kernel_ms * 1e-3) / 1e12
    print(json.dumps({
        "metric": METRIC, "value": K * T / (ms * 1e-3), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32+bf16x3", "data": "synthetic",
        "config": {"workload": "attn_qk", "which": "queries", "tokens": T, "draws": K,
                   "heads": H, "dv": 64, "d_in": c["d_in"], "seq_len": L, "sigma": c["sigma"],
                   "gamma": c["gamma"], "l2": "inputs larger than L2 (no flush)"},
        "roofline": {"bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                     "frac": ach / peak, "traffic": load_traffic({"name": "attn_qk"}),
                     "kernel": "attn_qk_tc_kernel<queries>", "kernel_ms": kernel_ms,
                     "flops": "algorithmic", "algorithmic_tflop": flops / 1e12,
                     "executed_tflop": executed / 1e12,
                     "peak_source": "bf16_tflops_sustained (%s)" % which},
        "cpu_baseline": None, "e2e": None, "gpu_launches": args.steps * 7,
        "clocks": clocks.summary()}), flush=True)
    return 0


def run_head_sweep(args):
    """The tiny head workload at K = 64 .. 16384: token-evals/s per K and the
    cosine of G_W with the analytic head gradient sum_t (softmax(z_t) -
    onehot(y_t)) x_t^T, next to the closed-form prediction 1/sqrt(1 + c/K)
    (the law cos(K) = c_max / sqrt(1 + c/K) the pages fit, Dust translation
    §4.2).  One JSON line per K."""
    import torch

    import activation_perturbation_es_noise_b300 as dust
    import workloads as W
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    p = W.HEAD_PARAMS["head_tiny"]
    wl = W.head_workload(p["T"], p["d"], p["V"], p["seq_len"], p["x_bf16"], p["zipf"])
    z64 = wl["z"].astype(np.float64)
    pr = np.exp(z64 - z64.max(1, keepdims=True))
    pr /= pr.sum(1, keepdims=True)
    g = pr.copy()
    g[np.arange(p["T"]), wl["targets"]] -= 1.0
    x64 = wl["x"].astype(np.float64)
    G = g.T @ x64
    c_pred = float(((x64 ** 2).sum(1) * (p["V"] + 1) * (g ** 2).sum(1)).sum() / (G ** 2).sum())
    zt = torch.from_numpy(wl["z"]).to(dev)
    yt = torch.from_numpy(wl["targets"]).to(dev)
    xt = torch.from_numpy(wl["x"]).to(dev)
    for K in W.HEAD_SWEEP_K:
        gh = torch.empty((p["T"], p["V"]), dtype=torch.float32, device=dev)
        Gw = torch.empty((p["V"], p["d"]), dtype=torch.float32, device=dev)
        ws = dust._workspace(dust.head_workspace_bytes(p["T"], p["V"], p["d"], K), dev)
        step = lambda: dust.head_estimate(zt, yt, xt, p["sigma"], K, W.NOISE_SEED, out=(gh, Gw),
                                          ws=ws)
        for _ in range(max(3, args.warmup)):
            step()
        torch.cuda.synchronize()
        # the inputs are far smaller than L2: flushed before every step
        ms = StepTimer(torch.cuda.current_stream(), True).time(args.steps, step) / args.steps
        Gk = Gw.double().cpu().numpy()
        cos = float((Gk * G).sum() / np.linalg.norm(Gk) / np.linalg.norm(G))
        print(json.dumps({"metric": METRIC, "value": K * p["T"] / (ms * 1e-3), "unit": UNIT,
                          "workload": "head_sweep", "draws": K, "ms_per_step": ms,
                          "cosine_vs_analytic": cos,
                          "cosine_predicted": 1.0 / np.sqrt(1.0 + c_pred / K),
                          "c_pred": c_pred}), flush=True)
    return 0


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    wl = make_workload(args.workload, "cpu", 0)
    for _ in range(args.warmup):
        pass  # the oracle has no warm-up state; its first call builds the C library
    import oracle
    oracle.lib()
    vals, sample = [], ""
    t0 = time.perf_counter()
    for _ in range(args.steps):
        v, sample = oracle_sample(wl, budget_s=max(2.0, 60.0 / max(args.steps, 1)))
        vals.append(v)
    elapsed = time.perf_counter() - t0
    value = float(np.median(vals))
    cores = os.cpu_count()
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * elapsed / max(args.steps, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference", "config": config_of(wl, args.gpus),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


def run_dust(args):
    import torch
    import torch.distributed as dist

    import activation_perturbation_es_noise_b300 as dust
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    dust.lib()
    wl = make_workload(args.workload, device, rank)
    estimate, evals, launches, ws, G_out = make_step(wl, dust)

    def step():
        # one estimator call, then the step's one exchange (N > 1): the sum of
        # the ranks' weight gradients
        estimate()
        if world > 1:
            dust.sum_over_ranks(G_out)
    for _ in range(max(args.warmup, 3 if args.warmup >= 3 else args.warmup)):
        step()
    torch.cuda.synchronize()
    if dust.workspace_status(ws) != 0:
        raise SystemExit("kernel status word set during warm-up")

    stream = torch.cuda.current_stream()
    timed = StepTimer(stream, l2_mode(wl) == "flush")
    barrier()
    with ClockSampler(local) as clocks:
        # the sampler's start leaves the GPU idle for 0.3 s: a few untimed steps
        # bring the clocks back up before the timed region
        for _ in range(max(3, args.warmup)):
            step()
        barrier()
        ms = timed.time(args.steps, step)
    barrier()
    # The dominant kernel's launches, timed in a second pass of the same steps
    # by events the library records around them on their stream (kept out of
    # the timed region above, where they would add host work per launch).
    timer = dust.KernelTimer(capacity=max(1, args.steps) * 64)
    with timer:
        # A bounded spin (about 0.5 ms per step) first, so that the host has
        # queued the steps' launches before the GPU reaches them: the events
        # then bracket the kernel alone, not host gaps between small launches.
        torch.cuda._sleep(1_000_000 * max(1, args.steps))
        for _ in range(args.steps):
            timed.flush()
            step()
    torch.cuda.synchronize()
    kernel_ms = timer.total_ms() / max(args.steps, 1)
    split = None
    if wl["kind"] == "interior":
        split = interior_kernel_split(timer.times_ms(), max(args.steps, 1))
        if split[1] is not None:
            kernel_ms = split[1]
        else:
            split = None
    if dust.workspace_status(ws) != 0:
        raise SystemExit("kernel status word set during the timed steps")
    ms_max = max_over_ranks(ms, dist if world > 1 else None)
    probes = issue_probes(dust) if wl["kind"] == "head" and rank == 0 else None

    # Optional: the same step captured once in a CUDA graph and replayed, which
    # removes the host's launch gaps between the call's kernels.
    graph = None
    if args.graph:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        stream.wait_stream(side)
        # one graph per input set when the steps rotate over copies
        graphs = []
        for _ in range(wl.get("rotate", 1)):
            graphs.append(torch.cuda.CUDAGraph())
            with torch.cuda.graph(graphs[-1]):
                step()
        for cg in graphs:
            cg.replay()
        torch.cuda.synchronize()
        nxt = [0]

        def replay():
            graphs[nxt[0]].replay()
            nxt[0] = (nxt[0] + 1) % len(graphs)
        gms = timed.time(args.steps, replay) / args.steps
        graph = {"ms_per_step": gms, "value": evals * world / (gms * 1e-3), "unit": UNIT}
    value = evals * world * args.steps / (ms_max * 1e-3)

    # End to end through the public API from pinned host buffers: the step's
    # inputs copied in, the estimator, the weight gradient copied out.
    # End to end through the public API from pinned host buffers: each step
    # copies its inputs in, runs the estimator and copies G_W back.  The
    # copies of step i + 1 run on a second stream into a second set of device
    # buffers while step i computes, as a batch stream would be fed.
    e2e = None
    if not args.no_e2e:
        bf = torch.bfloat16
        as_bf16 = {"interior": ("x", "W2", "W_head"), "head": ("x",) if wl.get("x_bf16") else (),
                   "embed": ()}[wl["kind"]]
        host = {}
        for k, v in wl["host"].items():
            t = torch.from_numpy(np.ascontiguousarray(v))
            host[k] = (t.to(bf) if k in as_bf16 else t).pin_memory()
        sets = [{k: torch.empty(v.shape, dtype=v.dtype, device=device) for k, v in host.items()}
                for _ in range(2)]
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        if wl["kind"] == "head":
            T, V, dd, K = wl["T"], wl["V"], wl["d"], wl["K"]
            g = torch.empty((T, V), dtype=torch.float32, device=device)
            G = torch.empty((V, dd), dtype=torch.float32, device=device)
            wse = dust._workspace(dust.head_workspace_bytes(T, V, dd, K), device)

            if wl["vchunk"]:
                wse = dust._workspace(dust.lib().dust_head_chunked_workspace(
                    T, V, dd, K, wl["vchunk"]), device)

            def call(d):
                if wl["vchunk"]:
                    dust.head_estimate_chunked(d["logits"], d["targets"], d["x"], wl["sigma"], K,
                                               1234, wl["vchunk"], token0=wl["token0"],
                                               out=(g, G), ws=wse)
                    return
                dust.head_estimate(d["logits"], d["targets"], d["x"], wl["sigma"], K, 1234, 0, 0,
                                   wl["token0"], out=(g, G), ws=wse, baseline=wl["baseline"])
        elif wl["kind"] == "interior":
            T, K = wl["T"], wl["K"]
            g = torch.empty((T, wl["C"]), dtype=torch.float32, device=device)
            G = torch.empty((wl["C"], wl["d_in"]), dtype=torch.float32, device=device)
            wse = dust._workspace(dust.linear_workspace_bytes(
                T, wl["d_in"], wl["C"], wl["d_model"], wl["V"], K), device)

            def call(d):
                dust.linear_estimate(d["x"], d["y1"], d["W2"], wl["lam"], d["W_head"],
                                     d["z_clean"], d["targets"], wl["seq_len"], wl["sigma"],
                                     wl["gamma"], K, 1234, 1, 0, wl["token0"], out=(g, G),
                                     ws=wse)
        else:
            V, dd, T = wl["V"], wl["d"], wl["T"]
            G = torch.empty((V, dd), dtype=torch.float32, device=device)
            perm = torch.empty(T, dtype=torch.int32, device=device)
            wse = dust._workspace(dust.embed_workspace_bytes(T, dd, V), device)

            def call(d):
                dust.embed_scatter(d["g"], d["ids"], V, out=(G, perm), ws=wse)
        estimate_call = call

        def call(d):
            estimate_call(d)
            if world > 1:
                dust.sum_over_ranks(G)
        Gh = torch.empty(G.shape, dtype=torch.float32).pin_memory()
        d2h = Gh.numel() * 4
        copy_s = torch.cuda.Stream(device=device)
        used = [torch.cuda.Event() for _ in range(2)]
        copied = [torch.cuda.Event() for _ in range(2)]

        def copy_in(b):
            with torch.cuda.stream(copy_s):
                copy_s.wait_event(used[b])
                for k in host:
                    sets[b][k].copy_(host[k], non_blocking=True)
                copied[b].record(copy_s)

        def run(n, start_event=None):
            if start_event is not None:
                copy_s.wait_event(start_event)
            copy_in(0)
            for i in range(n):
                if i + 1 < n:
                    copy_in((i + 1) % 2)
                stream.wait_event(copied[i % 2])
                call(sets[i % 2])
                used[i % 2].record(stream)
                Gh.copy_(G, non_blocking=True)

        run(max(2, args.warmup))
        torch.cuda.synchronize()
        barrier()
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        run(args.steps, f0)
        f1.record(stream)
        f1.synchronize()
        barrier()
        te = max_over_ranks(f0.elapsed_time(f1), dist if world > 1 else None)
        e2e = {"value": evals * world * args.steps / (te * 1e-3), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "overlap": "inputs of step i+1 copied on a second stream during step i"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, sample = oracle_sample(wl)
        cpu = {"value": v, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
               "sample": sample}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f32" if wl["kind"] != "interior" else "f32+bf16x2",
                "data": "synthetic", "config": config_of(wl, world),
                "roofline": roofline(wl, kernel_ms, load_traffic(wl), probes, split),
                "cpu_baseline": cpu, "e2e": e2e, "graph": graph,
                "gpu_launches": launches * args.steps,
                "clocks": clocks.summary()}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="dust", choices=["dust", "reference"])
    ap.add_argument("--workload", default="head_batch",
                    choices=["head_batch", "head_batch_antithetic", "head_batch_chunked",
                             "head_tiny", "head_scale",
                             "interior",
                             "interior_scale", "embed_scale", "head_sweep", "optim_adam",
                             "attn_value", "attn_qk"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="also time the step captured in a CUDA graph")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "head_sweep":
        return run_head_sweep(args)
    if args.workload == "optim_adam":
        return run_optim(args)
    if args.workload == "attn_value":
        return run_attn_value(args)
    if args.workload == "attn_qk":
        return run_attn_qk(args)
    return run_dust(args)


if __name__ == "__main__":
    sys.exit(main())
