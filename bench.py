"""Benchmark of the quantized speculative-decoding hot path on one GB300.

One step = one pass of the hot path over the 7B-class verify workload:
the 28-layer Qwen2.5-7B-shaped stack of W4A16 linears (q/o 3584x3584,
k/v 3584x512, gate/up 3584x18944, down 18944x3584, INT4 group 128) at
M = batch * (gamma + 1) = 5, followed by the speculative-sampling
verification over vocab 152064 (gamma 4, batch 1, T 1, target = draft +
N(0, sigma^2)).  Attention, norms, embedding and lm_head are not part of the
path and are not run.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0).  `value` is the algorithmic HBM GB/s of the
whole step (every packed weight byte, scale, zero, activation and output of
the stack, plus one read of every logit) over the device-timed step; the
`roofline` object reports the W4A16 GEMV (the dominant kernel) alone.
Inputs are resident in HBM before the timed region; `e2e` repeats the step
through the C ABI with the step's inputs copied from pinned host memory and
its result read back inside the timed region.

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the path needs no exchange between GPUs); value = total bytes of all ranks /
the slowest rank's time.
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
sys.path.insert(0, ROOT)

METRIC = "W4A16 GEMM HBM GB/s (% of roofline); spec-verify tokens/s at γ=4, 1 GB300"
WORKLOAD = "qwen7b"
SIGMA = 0.7


# ------------------------------------------------------------------ helpers
def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _gemm_bytes(M, N, K):
    """Algorithmic bytes of one W4A16 linear: int4 weights, fp16 scale and zero
    per group of 128, bf16 x in, bf16 y out."""
    return N * K // 2 + 4 * N * (K // 128) + 2 * M * K + 2 * M * N


def _verify_bytes(B, gamma, V):
    return 4 * B * (2 * gamma + 1) * V


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the run."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.gpu = gpu_index
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.perf_counter(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        win = [p for t, p in self.samples if t0 <= t <= t1]
        if not win:  # timed region shorter than the sampling period: nearest samples
            win = [p for t, p in self.samples if t0 - 0.3 <= t <= t1 + 0.3]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        sm = [num(p[1]) for p in win if num(p[1]) is not None]
        mx = [num(p[2]) for p in win if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in win for i in range(4) if p[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(win)}


def _traffic_record(src_hash):
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    if rec.get("kernel_source_sha256") != src_hash:
        return None
    return rec


def _kernel_source_hash():
    """Hash of the dominant kernel's code: w4a16_mma.cu and the device headers
    it includes.  A traffic record taken on other code for that kernel is not
    reported."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "quantized_speculative_decoding_gb300", "csrc")
    for name in ("w4a16_mma.cu", "device_common.cuh", "launch.cuh"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()


# ------------------------------------------------------------- oracle legs
def _oracle_sample(rows_per_shape: int, inputs):
    """The CPU oracle on a bounded sample of one step: `rows_per_shape` output
    rows of each of the 7 linears of one layer at M = 5, each linear timed on
    its own, and the full verification.  Returns ({linear: seconds per output
    row}, verify seconds, seconds of the whole sample)."""
    import oracle
    xs, packed, dl, tl, dt = inputs
    per_row = {}
    t_all = time.perf_counter()
    for (name, K, N), (qw, s, z) in zip(_layer(), packed):
        r = min(rows_per_shape, N)
        t0 = time.perf_counter()
        oracle.w4a16_linear(xs[K], qw[:r], s[:r], z[:r], 128, r, K)
        per_row[name] = (time.perf_counter() - t0) / r
    t0 = time.perf_counter()
    oracle.verify(dl, tl, dt, 4, 1.0, 0)
    t_verify = time.perf_counter() - t0
    return per_row, t_verify, time.perf_counter() - t_all


def _step_bytes():
    """Algorithmic bytes of one step, as the GPU line counts them: the 28 fused
    layers' linears at M = 5 and one read of every logit."""
    from quantized_speculative_decoding_gb300 import synth
    wl = synth.WORKLOADS[WORKLOAD]
    fused = [(K, N) for _, K, N, _ in synth.fused_layer(wl["layer"])]
    return (wl["layers"] * sum(_gemm_bytes(wl["M"], N, K) for K, N in fused) +
            _verify_bytes(wl["batch"], wl["gamma"], wl["vocab"]))


def _oracle_step_seconds(per_row, t_verify):
    """The oracle's time for a whole step, extrapolated from the sample: every
    output row of every linear of the 28 layers at its measured time per row,
    plus one verification."""
    from quantized_speculative_decoding_gb300 import synth
    wl = synth.WORKLOADS[WORKLOAD]
    return wl["layers"] * sum(N * per_row[name] for name, K, N in _layer()) + t_verify


def _layer():
    from quantized_speculative_decoding_gb300 import synth
    return synth.WORKLOADS[WORKLOAD]["layer"]


def _oracle_inputs(max_rows: int):
    """Host inputs for the oracle legs: max_rows rows of each layer-0 linear
    (drawn from the weight distribution for just those rows, so that many
    processes can hold a sample at once; packed by the oracle's own
    quantiser), the activations and the verify logits."""
    import oracle
    from quantized_speculative_decoding_gb300 import synth
    wl = synth.WORKLOADS[WORKLOAD]
    packed = []
    xs = {}
    for i, (name, K, N) in enumerate(wl["layer"]):
        r = min(max_rows, N)
        w = synth.weights(r, K, synth.weight_seed(wl["config"], 0, i))
        q, s, z = oracle.quantize_w4(w, 128)
        qw = np.bitwise_or.reduce(q.astype(np.uint32).reshape(r, K // 8, 8)
                                  << (4 * np.arange(8, dtype=np.uint32)), axis=2).astype(np.uint32)
        packed.append((qw, s, z))
        xs.setdefault(K, synth.activations(wl["M"], K))
    dl, tl = synth.logits(1, wl["gamma"], wl["vocab"], SIGMA, 11 + wl["config"])
    dt = synth.draft_tokens(dl, wl["T"], 11 + wl["config"])
    return xs, packed, dl, tl, dt


def _mean_rates(samples):
    """Per-row times and verify time averaged over samples (lists of
    _oracle_sample results)."""
    names = samples[0][0].keys()
    per_row = {n: float(np.mean([s[0][n] for s in samples])) for n in names}
    return per_row, float(np.mean([s[1] for s in samples]))


def cpu_baseline(budget_s: float = 20.0):
    """The oracle as it stands, single-threaded, timed on a bounded sample of
    the step (about budget_s seconds) and extrapolated to the whole step."""
    per16, tv, _ = _oracle_sample(16, _oracle_inputs(16))
    row_set = sum(per16.values())                 # seconds for one row of each linear
    rows = int(min(3584, max(16, (budget_s / 2 - tv) / max(row_set, 1e-9))))
    inputs = _oracle_inputs(rows)
    samples, t = [], 0.0
    while len(samples) < 4 and (not samples or t < 0.6 * budget_s):
        sm = _oracle_sample(rows, inputs)
        samples.append(sm)
        t += sm[2]
    per_row, t_verify = _mean_rates(samples)
    step_s = _oracle_step_seconds(per_row, t_verify)
    return {"value": _step_bytes() / step_s / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{len(samples)} x ({rows} output rows of each of the 7 W4A16 linears of one layer at M=5, "
                      f"each timed, plus the full V=152064 verify), {t:.1f} s single-threaded fp64; "
                      f"extrapolated to the whole step ({step_s:.1f} s: every row of the 28 layers at its "
                      f"measured time per row, plus one verify)",
            "extrapolated_step_s": step_s}


def _oracle_core_worker(rows, budget_s, barrier, results):
    """One host core's share of the all-cores leg: its own copy of the sample
    (built before the barrier, untimed), then oracle samples for budget_s."""
    try:
        inputs = _oracle_inputs(rows)
        barrier.wait(timeout=120)
        samples, t = [], 0.0
        while t < budget_s:
            sm = _oracle_sample(rows, inputs)
            samples.append(sm)
            t += sm[2]
        per_row, t_verify = _mean_rates(samples)
        results.put((_oracle_step_seconds(per_row, t_verify), len(samples)))
    except Exception as e:  # reported to the parent at once
        results.put(("error", f"{type(e).__name__}: {e}"))


def cpu_baseline_all_cores(budget_s: float = 10.0, cores: int = 0, rows: int = 64):
    """The oracle as it stands on every host core at once: each core runs its
    own copy of the bounded sample repeatedly, all started together, and
    extrapolates its own whole-step time; the rate is the step bytes of all
    cores over the slowest core's step time.  Worker processes are spawned,
    so this is safe whether or not CUDA is initialised."""
    import multiprocessing as mp
    n = cores or min(os.cpu_count() or 1, 16)
    ctx = mp.get_context("spawn")
    barrier, results = ctx.Barrier(n), ctx.Queue()
    procs = [ctx.Process(target=_oracle_core_worker, args=(rows, budget_s, barrier, results)) for _ in range(n)]
    for p_ in procs:
        p_.start()
    try:
        # bounded: a worker that dies (e.g. out of memory) must not hang the bench
        got = []
        for _ in range(n):
            r = results.get(timeout=budget_s + 180)
            if r[0] == "error":
                raise RuntimeError(r[1])
            got.append(r)
    finally:
        for p_ in procs:
            p_.join(timeout=30)
            if p_.is_alive():
                p_.terminate()  # only the processes started above
    step_s = max(g[0] for g in got)
    return {"value": n * _step_bytes() / step_s / 1e9, "unit": "GB/s", "cores": n, "kind": "oracle",
            "sample": f"{n} processes, each repeating ({rows} output rows of each of the 7 W4A16 linears of "
                      f"one layer at M=5, each timed, plus the full V=152064 verify) for about {budget_s:.0f} s "
                      f"and extrapolating its whole-step time; all processes' step bytes over the slowest "
                      f"one's step time ({step_s:.1f} s), fp64",
            "extrapolated_step_s": step_s}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    steps, warmup = args.steps, args.warmup
    inputs = _oracle_inputs(64)
    _, _, t4 = _oracle_sample(4, inputs)
    # samples sized so that the whole run takes about two minutes
    rows = int(max(2, min(64, 4 * (120.0 / max(1, steps + warmup)) / max(t4, 1e-6))))
    for _ in range(warmup):
        _oracle_sample(rows, inputs)
    step_s = []
    for _ in range(steps):
        per_row, t_verify, _ = _oracle_sample(rows, inputs)
        step_s.append(_oracle_step_seconds(per_row, t_verify))
    mean_s = float(np.mean(step_s))
    value = _step_bytes() / mean_s / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1,
        "steps": steps, "warmup": warmup, "ms_per_step": 1e3 * mean_s,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": _config(),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"per step: {rows} output rows of each of the 7 linears of one layer at "
                                   f"M=5, each timed, plus the full V=152064 verify; extrapolated to the "
                                   f"whole step (every row of the 28 layers at its measured time per row, "
                                   f"plus one verify)"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _config():
    return {"workload": "qwen7b-verify: 28 layers x {q,k,v,o 3584x3584/512, gate,up 3584x18944, "
                        "down 18944x3584} W4A16 g128 at M=5, then verify V=152064 gamma=4 B=1 T=1 "
                        f"sigma={SIGMA}",
            "packing": "q|k|v and gate|up concatenated along N (4 launches per layer)",
            "M": 5, "layers": 28, "vocab": 152064, "gamma": 4, "batch": 1, "sigma": SIGMA,
            "l2": "no flush: each step streams 3.47 GB of packed weights (>> 129 MB L2)"}


TRIALS = 128


def _acceptance_summary(lens, dl, tl, T):
    """Measured acceptance over independent trials (lens [trials][B], accepted
    draft tokens per trial) beside its closed form.  With x_i ~ q_i the chance
    that position i is accepted, given that every earlier one was, is
    beta_i = sum_x min(p_i(x), q_i(x)) (p, q the target and draft
    distributions at temperature T, in fp64); the expected number of emitted
    tokens is 1 + sum_{i=1..gamma} prod_{j<=i} beta_j.  The closed form holds
    for T > 0 only."""
    trials, B = lens.shape
    gamma = dl.shape[1]
    emitted = (lens + 1).sum(axis=1)            # tokens emitted by the batch per trial
    pos = [float((lens >= i + 1).mean()) for i in range(gamma)]
    cond = [float((lens >= i + 1).sum() / max(1, (lens >= i).sum())) for i in range(gamma)]
    out = {"trials": int(trials), "mean_emitted_tokens": float(emitted.mean()),
           "stderr_emitted_tokens": float(emitted.std(ddof=1) / np.sqrt(trials)) if trials > 1 else None,
           "position_acceptance": pos, "conditional_acceptance": cond,
           "draws": "each trial draws its own draft tokens (Gumbel-max from the draft distribution) "
                    "and uses its own Philox seed"}
    if T > 0:
        def softmax(a):
            a = a.astype(np.float64) / T
            e = np.exp(a - a.max(axis=-1, keepdims=True))
            return e / e.sum(axis=-1, keepdims=True)
        beta = np.minimum(softmax(tl[:, :gamma]), softmax(dl)).sum(axis=-1)   # [B][gamma]
        expected = (1.0 + np.cumprod(beta, axis=1).sum(axis=1)).sum()
        out["closed_form"] = {"beta": beta.mean(axis=0).tolist(),
                              "expected_emitted_tokens": float(expected),
                              "z": float((emitted.mean() - expected) / out["stderr_emitted_tokens"])
                              if out["stderr_emitted_tokens"] else None}
    return out


# --------------------------------------------------------------- GPU arm
def run_ours(args):
    import torch
    import torch.distributed as dist

    from quantized_speculative_decoding_gb300 import binding as sd
    from quantized_speculative_decoding_gb300 import replicas, synth

    world, rank, local = replicas.world_rank_local()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    wl = synth.WORKLOADS[WORKLOAD]
    M, L, V, gamma, B = wl["M"], wl["layers"], wl["vocab"], wl["gamma"], wl["batch"]
    # q/k/v and gate/up read the same x: each group is one packed matrix
    layer = [(name, K, N) for name, K, N, _ in synth.fused_layer(wl["layer"])]
    members = [idx for _, _, _, idx in synth.fused_layer(wl["layer"])]

    # ---- weights: layer 0 packed on the host (sd_w4_pack), put into the tiled
    # layout on the device (sd_w4_tile), copied to 28 distinct buffers
    base = []
    for i, (name, K, N) in enumerate(layer):
        w = np.concatenate([synth.weights(wl["layer"][j][2], K, synth.weight_seed(wl["config"], 0, j))
                            for j in members[i]])
        qw = np.zeros((N, K // 8), np.uint32)
        s = np.zeros((N, K // 128), np.uint16)
        z = np.zeros((N, K // 128), np.uint16)
        sd.sd_w4_pack(w, N, K, 128, qw, s, z)
        del w
        rowmajor = tuple(torch.from_numpy(a.view(np.int32) if a.dtype == np.uint32 else
                                          a.view(np.int16)).to(dev) for a in (qw, s, z))
        qb, sb = sd.sd_w4_tiled_bytes(N, K, 128)
        tiled = (torch.empty(qb, dtype=torch.uint8, device=dev),
                 torch.empty(sb // 2, dtype=torch.int16, device=dev))
        sd.sd_w4_tile(*rowmajor, 128, N, K, *tiled)
        base.append(tiled)
    torch.cuda.synchronize()
    weights = [[tuple(t.clone() for t in base[i]) for i in range(len(layer))] for _ in range(L)]
    torch.cuda.synchronize()
    del base
    xs = {K: torch.from_numpy(synth.activations(M, K).view(np.int16)).to(dev)
          for K in sorted({K for _, K, _ in layer})}
    outs = [[torch.empty((M, N), dtype=torch.bfloat16, device=dev) for (_, _, N) in layer]
            for _ in range(L)]
    dl, tl = synth.logits(B, gamma, V, SIGMA, 11 + wl["config"])
    dt = synth.draft_tokens(dl, wl["T"], 11 + wl["config"])
    d_dl = torch.from_numpy(dl).to(dev)
    d_tl = torch.from_numpy(tl).to(dev)
    d_dt = torch.from_numpy(dt).to(dev)
    out_tok = torch.empty((B, gamma + 1), dtype=torch.int32, device=dev)
    out_len = torch.empty((B,), dtype=torch.int32, device=dev)

    stream = torch.cuda.Stream(device=dev)

    def stack():
        for l in range(L):
            for i, (name, K, N) in enumerate(layer):
                tq, tsz = weights[l][i]
                sd.sd_w4a16_linear_tiled(xs[K], tq, tsz, 128, M, N, K, outs[l][i], stream)

    def verify(seed=0):
        sd.sd_verify(d_dl, d_tl, d_dt, gamma, B, V, wl["T"], seed, out_tok, out_len, stream)

    with torch.cuda.stream(stream):
        stack()
        verify()
    stream.synchronize()
    assert sd.sd_device_error(stream) == 0

    # emitted tokens per step over TRIALS independent trials (outside the
    # timing): each trial draws its own draft tokens x_i ~ q_i and runs the
    # verify with its own Philox seed; checked against the closed form
    lens = []
    for trial in range(TRIALS):
        d_dt.copy_(torch.from_numpy(synth.draft_tokens(dl, wl["T"], 20_000 + trial)))
        verify(trial)
        lens.append(out_len.cpu().numpy().copy())
    d_dt.copy_(torch.from_numpy(dt))
    stream.synchronize()
    lens = np.array(lens)                       # [TRIALS][B]
    acceptance = _acceptance_summary(lens, dl, tl, wl["T"])
    mean_emitted = acceptance["mean_emitted_tokens"]

    g_stack = torch.cuda.CUDAGraph()
    g_verify = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_stack, stream=stream):
        stack()
    with torch.cuda.graph(g_verify, stream=stream):
        verify(0)
    n_gemv = L * len(layer)
    n_verify = 2 if wl["T"] > 0 else 1

    stack_bytes = L * sum(_gemm_bytes(M, N, K) for _, K, N in layer)
    verify_bytes = _verify_bytes(B, gamma, V)
    step_bytes = stack_bytes + verify_bytes

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            g_stack.replay()
            g_verify.replay()
    stream.synchronize()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    replicas.barrier(world)
    torch.cuda.synchronize()
    t_host0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for k in range(K):
            ev[k][0].record(stream)
            g_stack.replay()
            ev[k][1].record(stream)
            g_verify.replay()
            ev[k][2].record(stream)
    torch.cuda.synchronize()
    t_host1 = time.perf_counter()
    replicas.barrier(world)
    t_stack = sum(ev[k][0].elapsed_time(ev[k][1]) for k in range(K)) / 1e3
    t_verify = sum(ev[k][1].elapsed_time(ev[k][2]) for k in range(K)) / 1e3
    t_total = ev[0][0].elapsed_time(ev[K - 1][2]) / 1e3
    t_total, t_stack, t_verify = replicas.max_over_ranks([t_total, t_stack, t_verify], world, dev)
    clocks = sampler.summary(t_host0, t_host1) if sampler else None

    # ---- e2e: the step through the C ABI with host buffers
    h_x = {K: torch.from_numpy(synth.activations(M, K).view(np.int16)).pin_memory() for K in xs}
    h_dl = torch.from_numpy(dl).pin_memory()
    h_tl = torch.from_numpy(tl).pin_memory()
    h_dt = torch.from_numpy(dt).pin_memory()
    h_tok = torch.empty((B, gamma + 1), dtype=torch.int32).pin_memory()
    h_len = torch.empty((B,), dtype=torch.int32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in list(h_x.values()) + [h_dl, h_tl, h_dt])
    d2h = h_tok.numel() * 4 + h_len.numel() * 4
    ke = max(3, min(K, 50))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    for it in range(ke + 2):
        if it == 2:
            replicas.barrier(world)
            torch.cuda.synchronize()
            e0.record(stream)
        with torch.cuda.stream(stream):
            for Kx, t in h_x.items():
                xs[Kx].copy_(t, non_blocking=True)
            d_dl.copy_(h_dl, non_blocking=True)
            d_tl.copy_(h_tl, non_blocking=True)
            d_dt.copy_(h_dt, non_blocking=True)
            g_stack.replay()
            g_verify.replay()
            h_tok.copy_(out_tok, non_blocking=True)
            h_len.copy_(out_len, non_blocking=True)
        stream.synchronize()  # the host reads the step's result
    e1.record(stream)
    torch.cuda.synchronize()
    t_e2e = e0.elapsed_time(e1) / 1e3 / ke
    t_e2e = replicas.max_over_ranks([t_e2e], world, dev)[0]
    if sampler:
        sampler.stop()
    assert sd.sd_device_error(stream) == 0

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    peak, peak_kind = _peaks()
    step_t = t_total / K
    gemv_t = t_stack / K / n_gemv                 # average W4A16 launch
    achieved = stack_bytes / n_gemv / gemv_t / 1e9
    src_hash = _kernel_source_hash()
    traffic = _traffic_record(src_hash)
    line = {
        "metric": METRIC,
        "value": replicas.whole_job_rate(world, step_bytes, step_t) / 1e9,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": 1e3 * step_t,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int4xbf16->f32",
        "data": "synthetic",
        "config": _config(),
        "roofline": {
            "bound": "hbm", "kernel": f"w4a16 linear (28 layers x {len(layer)} launches, average launch)",
            "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)" if peak_kind == "measured"
            else "fallback 6.8 TB/s",
            "frac_of_8tbs_nominal": achieved / 8000.0,
            "traffic": traffic["dram_bytes_per_launch"] if traffic else None,
        },
        "verify": {"us_per_call": 1e6 * t_verify / K,
                   "GBps": verify_bytes / (t_verify / K) / 1e9,
                   "launches_per_call": n_verify},
        "stack": {"us": 1e6 * t_stack / K, "GBps": stack_bytes / (t_stack / K) / 1e9,
                  "bytes": stack_bytes, "launches": n_gemv},
        "tokens_per_s": replicas.whole_job_rate(world, mean_emitted, step_t),
        "mean_emitted_tokens": mean_emitted,
        "position_acceptance": acceptance["position_acceptance"],
        "acceptance": acceptance,
        "e2e": {"value": replicas.whole_job_rate(world, step_bytes, t_e2e) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": 1e3 * t_e2e, "tokens_per_s": replicas.whole_job_rate(world, mean_emitted, t_e2e)},
        "gpu_launches": K * (n_gemv + n_verify),
        "clocks": clocks,
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline()
        try:
            line["cpu_baseline_all_cores"] = cpu_baseline_all_cores()
        except Exception as e:  # the headline line is printed either way
            line["cpu_baseline_all_cores"] = {"unavailable": f"{type(e).__name__}: {e}"}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_case(args):
    """Small fixed workloads for ncu captures (not a bench line): a few
    launches of one kernel on inputs larger than L2 but a few GB at most."""
    import torch

    from quantized_speculative_decoding_gb300 import binding as sd
    from quantized_speculative_decoding_gb300 import synth
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    name = args.case
    if name.startswith("w4-") or name.startswith("w4t-"):
        # w4-<M> / w4t-<M>: two Qwen2.5-7B-shaped layers (248 MB packed) at M
        # rows, row-major (sd_w4a16_linear, 7 launches per layer) or tiled
        # (sd_w4a16_linear_tiled, 4 launches per layer as in the bench step)
        M = int(name.split("-")[1])
        tiled_case = name.startswith("w4t-")
        # the tiled case mirrors the bench step: q|k|v and gate|up packed as one matrix each
        groups = (synth.fused_layer(synth.QWEN7B_LAYER) if tiled_case else
                  [(n, K, N, (i,)) for i, (n, K, N) in enumerate(synth.QWEN7B_LAYER)])
        layer = [(n, K, N) for n, K, N, _ in groups]
        bufs = []
        for i, (_, K, N) in enumerate(layer):
            w = np.concatenate([synth.weights(synth.QWEN7B_LAYER[j][2], K, synth.weight_seed(1, 0, j))
                                for j in groups[i][3]])
            qw = np.zeros((N, K // 8), np.uint32)
            s_ = np.zeros((N, K // 128), np.uint16)
            z = np.zeros((N, K // 128), np.uint16)
            sd.sd_w4_pack(w, N, K, 128, qw, s_, z)
            t = tuple(torch.from_numpy(a.view(np.int32) if a.dtype == np.uint32 else a.view(np.int16)).to(dev)
                      for a in (qw, s_, z))
            if tiled_case:
                qb, sb = sd.sd_w4_tiled_bytes(N, K, 128)
                tt = (torch.empty(qb, dtype=torch.uint8, device=dev),
                      torch.empty(sb // 2, dtype=torch.int16, device=dev))
                sd.sd_w4_tile(*t, 128, N, K, *tt)
                torch.cuda.synchronize()
                t = tt
            bufs.append((K, N, t, tuple(x.clone() for x in t)))
        torch.cuda.synchronize()
        linear = sd.sd_w4a16_linear_tiled if tiled_case else sd.sd_w4a16_linear
        xs = {K: torch.from_numpy(synth.activations(M, K).view(np.int16)).to(dev) for _, K, _ in layer}
        out = {N: torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _, _, N in layer}
        for rep in range(3):
            for copy in (0, 1):
                for K, N, t0, t1 in bufs:
                    linear(xs[K], *(t0 if copy == 0 else t1), 128, M, N, K, out[N])
        torch.cuda.synchronize()
    elif name.startswith("lm-"):
        # lm-<M>: the 7B target's lm_head in logits mode (V = 152064, K = 3584,
        # 290 MB packed INT4) at M rows, two weight copies, T = 1, three rounds
        M, V, K = int(name.split("-")[1]), 152064, 3584
        copies = []
        for c in range(2):
            qw, s_, z = synth.packed_w4(V, K, 300 + c)
            t = tuple(torch.from_numpy(a.view(np.int32) if a.dtype == np.uint32 else a.view(np.int16)).to(dev)
                      for a in (qw, s_, z))
            qb, sb = sd.sd_w4_tiled_bytes(V, K, 128)
            tt = (torch.empty(qb, dtype=torch.uint8, device=dev), torch.empty(sb // 2, dtype=torch.int16, device=dev))
            sd.sd_w4_tile(*t, 128, V, K, *tt)
            torch.cuda.synchronize()
            copies.append(tt)
            del t
        parts = sd.sd_lm_head_parts(M, V, K)
        x = torch.from_numpy(synth.activations(M, K).view(np.int16)).to(dev)
        logits = torch.empty((M, V), dtype=torch.float32, device=dev)
        stats = torch.empty((M, parts, 2), dtype=torch.float32, device=dev)
        for rep in range(3):
            for tt in copies:
                sd.sd_w4a16_lm_head(x, *tt, 128, M, V, K, 1.0, logits, V, stats, parts)
        torch.cuda.synchronize()
    elif name == "verify":
        wl = synth.WORKLOADS["qwen7b"]
        B = 8  # 8 x 9 rows x 152064 = 43.8 MB per call; 4 distinct input sets > L2
        sets = []
        for i in range(4):
            dl, tl = synth.logits(B, 4, wl["vocab"], SIGMA, 100 + i)
            dt = synth.draft_tokens(dl, 1.0, 100 + i)
            sets.append(tuple(torch.from_numpy(a).to(dev) for a in (dl, tl, dt)))
        tok = torch.empty((B, 5), dtype=torch.int32, device=dev)
        alen = torch.empty((B,), dtype=torch.int32, device=dev)
        for rep in range(2):
            for dl, tl, dt in sets:
                sd.sd_verify(dl, tl, dt, 4, B, wl["vocab"], 1.0, rep, tok, alen)
        torch.cuda.synchronize()
    else:
        raise SystemExit(f"unknown case {name}")
    print(f"case {name} done")
    return 0


# --------------------------------------------------------------- row sweep
def run_sweep(args):
    """One JSON line per measurement of the other rows of the path: the tiled
    W4A16 kernel per shape at M = 1..7 (7B fused shapes, 4B gamma sweep), the
    batched row-major W4A16 at M = 40/80/160 (Llama-7B shapes), the M = 1
    draft linears in bf16 / INT8 / INT4 (1.5B shapes, per shape and as a
    28-layer stack) and the verify at every workload's (B, gamma, V, T).
    Every timing replays a CUDA graph over enough distinct input copies to
    exceed L2; nothing here is the headline line."""
    import torch

    from quantized_speculative_decoding_gb300 import binding as sd
    from quantized_speculative_decoding_gb300 import synth
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    st = torch.cuda.Stream()
    peak, _ = _peaks()
    tf_peak = _tensor_peak()
    big = 320e6  # bytes of distinct inputs per measurement (> 2x L2)
    rows = set(args.rows.split(","))

    def gtime(calls, replays=10):
        with torch.cuda.stream(st):
            for c in calls:
                c()
        st.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            for c in calls:
                c()
        with torch.cuda.stream(st):
            for _ in range(3):
                g.replay()
        st.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(st):
            e0.record(st)
            for _ in range(replays):
                g.replay()
            e1.record(st)
        st.synchronize()
        return e0.elapsed_time(e1) * 1e3 / (replays * len(calls))  # us per call

    def emit(**kw):
        print(json.dumps(kw), flush=True)

    def dev16(a):
        return torch.from_numpy(a.view(np.int32) if a.dtype == np.uint32 else a.view(np.int16)).to(dev)

    def packed_w4(N, K, seed, tiled):
        w = synth.weights(N, K, seed)
        qw = np.zeros((N, K // 8), np.uint32)
        s_ = np.zeros((N, K // 128), np.uint16)
        z = np.zeros((N, K // 128), np.uint16)
        sd.sd_w4_pack(w, N, K, 128, qw, s_, z)
        t = tuple(dev16(a) for a in (qw, s_, z))
        if not tiled:
            return t
        qb, sb = sd.sd_w4_tiled_bytes(N, K, 128)
        tt = (torch.empty(qb, dtype=torch.uint8, device=dev), torch.empty(sb // 2, dtype=torch.int16, device=dev))
        sd.sd_w4_tile(*t, 128, N, K, *tt)
        torch.cuda.synchronize()
        return tt

    if "a2" in rows:
        # ---- a2: tiled W4A16 per shape
        shapes = [("7b." + n, K, N, 1) for n, K, N, _ in synth.fused_layer(synth.QWEN7B_LAYER)]
        shapes += [("4b." + n, K, N, 4) for n, K, N, _ in synth.fused_layer(synth.QWEN4B_LAYER)]
        for name, K, N, cfg in shapes:
            for layout in ("tiled", "row-major"):
                base = packed_w4(N, K, synth.weight_seed(cfg, 0, 0), layout == "tiled")
                nbytes = sum(a.numel() * a.element_size() for a in base)
                copies = [tuple(a.clone() for a in base) for _ in range(max(2, int(big // nbytes) + 1))]
                linear = sd.sd_w4a16_linear_tiled if layout == "tiled" else sd.sd_w4a16_linear
                for M in ((1, 3, 5, 7) if cfg == 1 else (3, 4, 5, 6, 7)):
                    x = torch.from_numpy(synth.activations(M, K).view(np.int16)).to(dev)
                    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
                    us = gtime([lambda c=c: linear(x, *c, 128, M, N, K, out, st) for c in copies])
                    b = _gemm_bytes(M, N, K)
                    emit(row="a2", kernel=f"w4a16 {layout} (mma.sync)", shape=name, K=K, N=N, M=M, us=us,
                         GBps=b / us / 1e3, frac=b / us / 1e3 / peak)
                del copies, base
                torch.cuda.empty_cache()

    if "a3" in rows:
        # ---- a3: batched row-major W4A16 (tcgen05) at M = 40 / 80 / 160
        for name, K, N in synth.LLAMA7B_LAYER[3:]:  # o (= q, k, v), gate (= up), down
            base = packed_w4(N, K, synth.weight_seed(3, 0, 0), False)
            nbytes = N * K // 2 + 4 * N * (K // 128)
            copies = [tuple(a.clone() for a in base) for _ in range(max(2, int(big // nbytes) + 1))]
            for M in (40, 80, 160):
                x = torch.from_numpy(synth.activations(M, K).view(np.int16)).to(dev)
                out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
                us = gtime([lambda c=c: sd.sd_w4a16_linear(x, *c, 128, M, N, K, out, st) for c in copies])
                b = _gemm_bytes(M, N, K)
                fl = 2.0 * M * N * K
                emit(row="a3", kernel="w4a16 row-major (tcgen05)", shape="llama7b." + name, K=K, N=N, M=M, us=us,
                     GBps=b / us / 1e3, frac_hbm=b / us / 1e3 / peak, TFLOPs=fl / us / 1e6,
                     frac_tensor=fl / us / 1e6 / tf_peak)
            del copies, base
            torch.cuda.empty_cache()

    if "a4" in rows:
        # ---- a4: M = 1 draft linears, 1.5B shapes: bf16 / INT8 / INT4 (row-major GEMV, tiled mma)
        layer = synth.QWEN1P5B_LAYER
        L = 28
        fmts = {}
        for fmt in ("bf16", "int8", "int4", "int4-tiled"):
            bufs = []
            for i, (n, K, N) in enumerate(layer):
                if fmt == "bf16":
                    w = torch.randn((N, K), device=dev).mul_(0.02).to(torch.bfloat16)
                    one = (w,)
                elif fmt == "int8":
                    one = (torch.randint(-127, 128, (N, K), dtype=torch.int8, device=dev),
                           torch.full((N,), 0x2000, dtype=torch.int16, device=dev))
                else:
                    one = packed_w4(N, K, synth.weight_seed(2, 0, i), fmt == "int4-tiled")
                bufs.append(one)
            fmts[fmt] = [[tuple(a.clone() for a in b) for b in bufs] for _ in range(L)]
            del bufs
        xs = {K: torch.from_numpy(synth.activations(1, K).view(np.int16)).to(dev) for _, K, _ in layer}
        outs = {N: torch.empty((1, N), dtype=torch.bfloat16, device=dev) for _, _, N in layer}

        def call(fmt, i, b):
            n, K, N = layer[i]
            if fmt == "bf16":
                return lambda: sd.sd_bf16_linear(xs[K], b[0], 1, N, K, outs[N], st)
            if fmt == "int8":
                return lambda: sd.sd_w8a16_linear(xs[K], b[0], b[1], 1, N, K, outs[N], st)
            if fmt == "int4":
                return lambda: sd.sd_w4a16_linear(xs[K], *b, 128, 1, N, K, outs[N], st)
            return lambda: sd.sd_w4a16_linear_tiled(xs[K], *b, 128, 1, N, K, outs[N], st)

        def wbytes(fmt, N, K):
            return {"bf16": 2 * N * K, "int8": N * K + 2 * N}.get(fmt, N * K // 2 + 4 * N * (K // 128)) + 2 * K + 2 * N

        for fmt, layers in fmts.items():
            for i, (n, K, N) in enumerate(layer):
                us = gtime([call(fmt, i, layers[l][i]) for l in range(L)])
                b = wbytes(fmt, N, K)
                emit(row="a4", kernel=fmt, shape="1.5b." + n, K=K, N=N, M=1, us=us, GBps=b / us / 1e3,
                     frac=b / us / 1e3 / peak)
            calls = [call(fmt, i, layers[l][i]) for l in range(L) for i in range(len(layer))]
            us = gtime(calls, replays=5) * len(calls)
            b = L * sum(wbytes(fmt, N, K) for _, K, N in layer)
            emit(row="a4", kernel=fmt, shape="1.5b.stack(28 layers)", M=1, us=us, GBps=b / us / 1e3, frac=b / us / 1e3 / peak)
        del fmts
        torch.cuda.empty_cache()

    if "a5-a9" in rows:
        # ---- a5..a9: verify
        cases = [(1, 4, 152064, 1.0, 0.7), (1, 4, 152064, 0.0, 0.7)]
        cases += [(B, 4, 32000, 0.8, 0.7) for B in (8, 16, 32)]
        cases += [(1, g, 151936, T, 0.5) for g in (2, 3, 4, 5, 6) for T in (0.0, 1.0)]
        for B, gamma, V, T, sigma in cases:
            vb = _verify_bytes(B, gamma, V) if T > 0 else 4 * B * (gamma + 1) * V
            n = max(2, int(big // _verify_bytes(B, gamma, V)) + 1)
            sets = []
            for i in range(n):
                dl, tl = synth.logits(B, gamma, V, sigma, 100 + i) if i < 4 else (None, None)
                if i < 4:
                    dt = synth.draft_tokens(dl, T, 100 + i)
                    base = tuple(torch.from_numpy(a).to(dev) for a in (dl, tl, dt))
                sets.append(tuple(a.clone() for a in base))
            tok = torch.empty((B, gamma + 1), dtype=torch.int32, device=dev)
            alen = torch.empty((B,), dtype=torch.int32, device=dev)
            us = gtime([lambda s_=s_: sd.sd_verify(*s_, gamma, B, V, T, 0, tok, alen, st) for s_ in sets])
            emit(row="a5-a9", kernel="verify", B=B, gamma=gamma, V=V, T=T, us=us, GBps=vb / us / 1e3,
                 frac=vb / us / 1e3 / peak, tokens_per_s_verify_only=None)
            del sets
            torch.cuda.empty_cache()

    if "next-4" in rows:
        # ---- next: INT3 / INT2 tiled linears (7B fused shapes) and the W4A4 draft linear (1.5B shapes)
        def packed_wb(N, K, bits, seed):
            w = synth.weights(N, K, seed)
            packed = np.zeros((N, K * bits // 32), np.uint32)
            s_ = np.zeros((N, K // 128), np.uint16)
            z = np.zeros((N, K // 128), np.uint16)
            sd.sd_wb_pack(w, N, K, 128, bits, packed, s_, z)
            qb, sb = sd.sd_wb_tiled_bytes(N, K, bits)
            tt = (torch.empty(qb, dtype=torch.uint8, device=dev), torch.empty(sb // 2, dtype=torch.int16, device=dev))
            sd.sd_wb_tile(dev16(packed), dev16(s_), dev16(z), 128, bits, N, K, *tt)
            torch.cuda.synchronize()
            return tt

        fused7 = [(n, K, N) for n, K, N, _ in synth.fused_layer(synth.QWEN7B_LAYER)]
        for bits in (4, 3, 2):
            for name, K, N in fused7:
                base = packed_wb(N, K, bits, synth.weight_seed(1, 0, 0))
                nbytes = sum(a.numel() * a.element_size() for a in base)
                copies = [tuple(a.clone() for a in base) for _ in range(max(2, int(big // nbytes) + 1))]
                for M in (1, 5, 8):
                    x = torch.from_numpy(synth.activations(M, K).view(np.int16)).to(dev)
                    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
                    us = gtime([lambda c=c: sd.sd_wb_linear_tiled(x, *c, 128, bits, M, N, K, out, st)
                                for c in copies])
                    b = nbytes + 2 * M * K + 2 * M * N
                    emit(row="next-4", kernel=f"int{bits} tiled (mma.sync)", shape="7b." + name, K=K, N=N, M=M,
                         us=us, GBps=b / us / 1e3, frac=b / us / 1e3 / peak, weight_bits=bits)
                del copies, base
                torch.cuda.empty_cache()
        # W4A4 at M = 1 on the 1.5B draft shapes: the activation quantiser, the
        # linear on its codes, and both back to back
        for i, (name, K, N) in enumerate(synth.QWEN1P5B_LAYER):
            base = packed_w4(N, K, synth.weight_seed(2, 0, i), True)
            nbytes = sum(a.numel() * a.element_size() for a in base)
            copies = [tuple(a.clone() for a in base) for _ in range(max(2, int(big // nbytes) + 1))]
            x = torch.from_numpy(synth.activations(1, K).view(np.int16)).to(dev)
            qx = torch.empty((1, K), dtype=torch.bfloat16, device=dev)
            sx = torch.empty((1, K // 128), dtype=torch.float32, device=dev)
            out = torch.empty((1, N), dtype=torch.bfloat16, device=dev)
            sd.sd_a4_quantize(x, 1, K, qx, sx, st)
            us_lin = gtime([lambda c=c: sd.sd_w4a4_linear_tiled(qx, sx, *c, 128, 1, N, K, out, st) for c in copies])
            us_both = gtime([c_ for c in copies for c_ in (lambda: sd.sd_a4_quantize(x, 1, K, qx, sx, st),
                                                          lambda c=c: sd.sd_w4a4_linear_tiled(qx, sx, *c, 128, 1, N,
                                                                                              K, out, st))]) * 2
            b = nbytes + 2 * K + 2 * N
            emit(row="next-4", kernel="w4a4 tiled (mma.sync)", shape="1.5b." + name, K=K, N=N, M=1,
                 us_linear=us_lin, us_with_quantiser=us_both, GBps=b / us_lin / 1e3, frac=b / us_lin / 1e3 / peak)
            del copies, base
            torch.cuda.empty_cache()

    if "next-1" in rows:
        # ---- next: the lm_head in logits mode (fp32 logits + softmax partials), target M = 5
        # (7B, K = 3584) and draft M = 1 (1.5B, K = 1536) over V = 152064, then the verify
        # from those partials against the verify with its own statistics pass
        V, gamma, B = 152064, 4, 1
        heads = {}
        for tag, M, K, seed in (("target", B * (gamma + 1), 3584, 300), ("draft", B, 1536, 301)):
            qw, s_, z = synth.packed_w4(V, K, seed)
            base = tuple(dev16(a) for a in (qw, s_, z))
            qb, sb = sd.sd_w4_tiled_bytes(V, K, 128)
            tiled = (torch.empty(qb, dtype=torch.uint8, device=dev), torch.empty(sb // 2, dtype=torch.int16, device=dev))
            sd.sd_w4_tile(*base, 128, V, K, *tiled)
            torch.cuda.synchronize()
            del base
            nb = qb + sb
            copies = [tiled] + [tuple(a.clone() for a in tiled) for _ in range(int(big // nb))]
            parts = sd.sd_lm_head_parts(M, V, K)
            x = torch.from_numpy(synth.activations(M, K, seed=seed).view(np.int16)).to(dev)
            lg = torch.empty((M, V), dtype=torch.float32, device=dev)
            ps = torch.empty((M, parts, 2), dtype=torch.float32, device=dev)
            for T in (1.0, 0.0):
                us = gtime([lambda c=c: sd.sd_w4a16_lm_head(x, *c, 128, M, V, K, T, lg, V, ps, parts, st)
                            for c in copies])
                b = V * K // 2 + 4 * V * (K // 128) + 2 * M * K + 4 * M * V + 8 * M * parts
                emit(row="next-1", kernel="w4a16 lm_head (fp32 logits + softmax partials)", role=tag, M=M, V=V,
                     K=K, T=T, parts=parts, us=us, GBps=b / us / 1e3, frac=b / us / 1e3 / peak)
            heads[tag] = (copies[0], x, parts, K)
            del copies
            torch.cuda.empty_cache()
        # the verify's inputs as the lm_heads write them: target rows in one call,
        # draft step i into row (b, i) through the strides
        (tq, xt, pt, Kt), (dq, xd, pd, Kd) = heads["target"], heads["draft"]
        for T in (1.0, 0.0):
            n = max(2, int(big // _verify_bytes(B, gamma, V)) + 1)
            sets = []
            for i in range(n):
                tl = torch.empty((B, gamma + 1, V), dtype=torch.float32, device=dev)
                ts = torch.empty((B, gamma + 1, pt, 2), dtype=torch.float32, device=dev)
                dl = torch.empty((B, gamma, V), dtype=torch.float32, device=dev)
                ds = torch.empty((B, gamma, pd, 2), dtype=torch.float32, device=dev)
                sd.sd_w4a16_lm_head(xt, *tq, 128, B * (gamma + 1), V, Kt, T, tl, V, ts, pt)
                for j in range(gamma):
                    sd.sd_w4a16_lm_head(xd, *dq, 128, B, V, Kd, T, dl[:, j].data_ptr(), gamma * V,
                                        ds[:, j].data_ptr(), gamma * pd)
                torch.cuda.synchronize()
                dt = torch.from_numpy(synth.draft_tokens(dl.cpu().numpy(), T, 400 + i)).to(dev)
                sets.append((dl, tl, ds, ts, dt))
            tok = torch.empty((B, gamma + 1), dtype=torch.int32, device=dev)
            alen = torch.empty((B,), dtype=torch.int32, device=dev)
            us_parts = gtime([lambda q=q: sd.sd_verify_parts(q[0], q[1], q[2], pd, q[3], pt, q[4], gamma, B, V, T, 0,
                                                              tok, alen, st) for q in sets])
            us_full = gtime([lambda q=q: sd.sd_verify(q[0], q[1], q[4], gamma, B, V, T, 0, tok, alen, st)
                             for q in sets])
            emit(row="next-1", kernel="verify from lm_head partials vs verify with its statistics pass",
                 B=B, gamma=gamma, V=V, T=T, us_parts=us_parts, us_stats_pass=us_full,
                 saved_us=us_full - us_parts)
            del sets
            torch.cuda.empty_cache()
        del heads
        torch.cuda.empty_cache()

    if "next-2" in rows:
        # ---- next: the draft-side sampler (one read of the logits)
        for B, V, T in [(1, 152064, 1.0), (1, 152064, 0.0), (8, 32000, 0.8), (32, 32000, 0.8),
                        (32, 152064, 1.0)]:
            sb = 4 * B * V
            n = max(2, int(big // sb) + 1)
            rows = torch.from_numpy(synth.logits(B, 1, V, 0.7, 200)[0][:, 0].copy()).to(dev)
            sets = [rows.clone() for _ in range(n)]
            tok = torch.empty((B,), dtype=torch.int32, device=dev)
            us = gtime([lambda x=x: sd.sd_sample(x, B, V, T, 0, 0, tok, st) for x in sets])
            emit(row="next-2", kernel="sample", B=B, V=V, T=T, us=us, GBps=sb / us / 1e3,
                 frac=sb / us / 1e3 / peak)
            del sets
            torch.cuda.empty_cache()
    if "next-3" in rows:
        # ---- next: the draft-gamma-then-verify step as one CUDA graph (1.5B draft, 7B target)
        from quantized_speculative_decoding_gb300 import spec_step
        wl = synth.WORKLOADS["qwen7b"]
        target_w = spec_step.build_weights(synth.QWEN7B_LAYER, wl["layers"], 1, "int4-tiled", dev)
        for fmt, gammas in (("int4-tiled", (1, 2, 3, 4, 5, 6)), ("int8", (4,)), ("bf16", (4,))):
            draft_w = spec_step.build_weights(synth.QWEN1P5B_LAYER, 28, 2, fmt, dev)
            for gamma in gammas:
                step = spec_step.SpecStep(draft_layer=synth.QWEN1P5B_LAYER, draft_layers=28, draft_fmt=fmt,
                                          target_layer=synth.QWEN7B_LAYER, target_layers=wl["layers"],
                                          gamma=gamma, vocab=wl["vocab"], temperature=1.0, sigma=SIGMA,
                                          seed=11 + wl["config"], draft_weights=draft_w, target_weights=target_w)
                times = {}
                for part in ("step", "draft", "target"):
                    g = step.capture(part, 0, st)
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    with torch.cuda.stream(st):  # replay() launches on the current stream
                        for _ in range(3):
                            g.replay()
                        e0.record(st)
                        for _ in range(10):
                            g.replay()
                        e1.record(st)
                    st.synchronize()
                    times[part] = e0.elapsed_time(e1) * 1e3 / 10
                    del g
                lens = []
                for seed in range(32):
                    with torch.cuda.stream(st):
                        step.step(seed, st)
                    st.synchronize()
                    lens.append(int(step.accept_len.item()))
                emitted = 1.0 + float(np.mean(lens))
                emit(row="next-3", kernel="draft+verify step graph", draft=fmt, gamma=gamma,
                     us_step=times["step"], us_draft=times["draft"], us_target=times["target"],
                     draft_share=times["draft"] / (times["draft"] + times["target"]),
                     mean_emitted=emitted, tokens_per_s=emitted / times["step"] * 1e6,
                     draft_GBps=gamma * step.draft_weight_bytes() / times["draft"] / 1e3,
                     target_GBps=step.target_weight_bytes() / times["target"] / 1e3)
                del step
            del draft_w
            torch.cuda.empty_cache()
        del target_w
        torch.cuda.empty_cache()
    assert sd.sd_device_error(st) == 0
    return 0


def _tensor_peak():
    """Measured dense bf16 TFLOP/s (burst), else the fallback 1900."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["bf16_tflops"])
    except Exception:
        return 1900.0


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", default=None,
                    help="run a small fixed workload for profiling (w4-<M>, w4t-<M>, lm-<M>, verify) and exit")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="measure the other rows (per-shape W4A16, batched M, M=1 draft formats, verify) and exit")
    ap.add_argument("--rows", default="a2,a3,a4,a5-a9,next-1,next-2,next-3,next-4",
                    help="with --sweep: the rows to measure, comma-separated")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    return args


def main():
    args = parse_args()
    if args.case:
        return run_case(args)
    if args.sweep:
        return run_sweep(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
