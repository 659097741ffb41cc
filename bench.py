"""Benchmark of the DSpark draft/verify hot path on GB300.

One step = one pass of the whole hot path over one synthetic batch:
    dspark_draft_logits -> dspark_markov_sample_conf (the sampler with the calibrated confidence
    head inside it) -> dspark_verify -> dspark_schedule (on the head's confidences)
Metric: draft tokens per second (B*N drafted tokens per step), plus the roofline
fraction of the dominant kernel and of the Markov sampler.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--secondary NAME|none]
                  [--impl gpu|reference]

The default workload is the batched serving draft (B=64, N=16, r=256); the
single-request Qwen3-8B-shaped decode (B=1, N=8) is measured after it in the
same run and reported in the same JSON line under "secondary".

Under torchrun (N > 1) every rank runs its own replica of the workload on its own
GPU (requests shard across GPUs with no data exchange: weak scaling); ranks meet
only at the timing barriers.  `--impl reference` times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
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

from workloads import (DRAFT_CONFIGS, SCHEDULE_CONFIGS, VerifyConfig, ScheduleConfig, draft_inputs,  # noqa: E402
                       verify_inputs, schedule_inputs)

METRIC = "draft tokens/sec (B·N per draft step) and % of roofline for logits+Markov sampling"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 512 * 1024 * 1024      # > 4x the 129 MB L2
WORKLOAD_TEMPERATURE = {"qwen3_8b_single": 1.0, "batched_draft": 0.8, "tiny": 1.0}

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one dspark_draft_logits launch on
# each workload, from one ncu capture of that kernel on that workload, with a digest of the
# kernel's sources at capture time: once the sources change the figure is reported as null.
GEMM_TRAFFIC = {
    "qwen3_8b_single": {"bytes": 1244772416 + 3775872, "src_digest": "65d3d273941b"},
    "batched_draft": {"bytes": 1271540416 + 590384128, "src_digest": "65d3d273941b"},
}
GEMM_SOURCES = ("draft_sampling_verification_tcgen05_gb300/csrc/draft_logits.cu",
                "draft_sampling_verification_tcgen05_gb300/csrc/device_common.cuh")


def gemm_source_digest():
    import hashlib
    h = hashlib.sha256()
    for rel in GEMM_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]



def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="batched_draft", choices=sorted(DRAFT_CONFIGS))
    ap.add_argument("--secondary", default="qwen3_8b_single", choices=sorted(DRAFT_CONFIGS) + ["none"],
                    help="a second workload measured after the first (GPU figures only)")
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch the four calls eagerly each step")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="budget of the oracle sample")
    ap.add_argument("--oracle-one-request", action="store_true", help=argparse.SUPPRESS)
    return ap.parse_args()


# ---------------------------------------------------------------------------
# workload construction (host, seeded)
# ---------------------------------------------------------------------------
def step_configs(name: str):
    d = DRAFT_CONFIGS[name]
    v = VerifyConfig(f"{name}_verify", B=d.B, gamma=d.N, V=d.V, target_std=3.0,
                     draft_sigmas=(0.3, 1.0, 3.0), independent_draft=False,
                     data_seed=d.data_seed + 4)
    s = ScheduleConfig(f"{name}_schedule", B=d.B, N=d.N, K_in=-1,
                       beta_mix=((9, 1), (5, 2), (2, 3)), sps_len=d.B * d.N,
                       data_seed=d.data_seed + 5)
    return d, v, s


def head_weights(d):
    """Synthetic weights of the calibrated confidence head: w_h ~ N(0, 1/H), w_e ~ N(0, 1/r), beta 0.5,
    a calibration temperature per position uniform in [0.7, 1.6]."""
    hrng = np.random.default_rng(d.data_seed + 7)
    w_h = (hrng.standard_normal(d.H) / np.sqrt(d.H)).astype(np.float32)
    w_e = (hrng.standard_normal(d.r) / np.sqrt(d.r)).astype(np.float32)
    tau = hrng.uniform(0.7, 1.6, d.N).astype(np.float32)
    return w_h, w_e, 0.5, tau


def host_inputs(name: str):
    d, v, s = step_configs(name)
    di = draft_inputs(d)
    vi = verify_inputs(v)
    si = schedule_inputs(s)
    T = np.full(d.B, WORKLOAD_TEMPERATURE[name], np.float32)
    return d, v, s, di, vi, si, T


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
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
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        t0, t1 = getattr(self, "window", (-1e30, 1e30))
        inside = [ln for t, ln in self.lines if t0 - 0.25 <= t <= t1 + 0.25]
        for ln in inside or [ln for _, ln in self.lines]:
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
            except ValueError:
                continue
            for n, val in zip(names, p[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "samples_in_timed_region": len(inside)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
class Arena:
    """One allocation holding several tensors at 256-byte aligned offsets (device, or pinned host
    memory): a step's inputs (or outputs) then cross between host and device in one copy."""

    def __init__(self, specs, device=None, pin=False):
        import torch
        self.offsets, off = {}, 0
        for name, shape, dtype in specs:
            nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
            self.offsets[name] = (off, shape, dtype, nbytes)
            off = (off + nbytes + 255) & ~255
        self.nbytes = off
        self.buf = torch.empty(off, dtype=torch.uint8, device=device, pin_memory=pin)

    def view(self, name):
        off, shape, dtype, nbytes = self.offsets[name]
        return self.buf[off: off + nbytes].view(dtype).view(shape)


def _nvtx(name):
    """An NVTX range around one C-ABI call (host side; visible in a profiler's timeline)."""
    import contextlib
    import torch
    try:
        return torch.cuda.nvtx.range(name)
    except Exception:                             # a build without NVTX: no range
        return contextlib.nullcontext()


def _timed_calls(fn, flush_l2, stream, n=20):
    """Median CUDA-event time (ms) of `fn` over n launches, L2 flushed before each."""
    import torch
    for _ in range(3):
        fn()
    ms = []
    for k in range(n):
        flush_l2(k)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    return float(np.median(ms))


def measure(name, args, dev, dist, world, rank, full):
    """Time the step on workload `name`; with `full`, also the end-to-end leg, the library's
    other entry points and the oracle leg.  Returns the JSON fields of the line."""
    import torch
    import draft_sampling_verification_tcgen05_gb300 as ds
    from draft_sampling_verification_tcgen05_gb300.replicas import job_throughput, max_over_ranks, replica_seed
    from workloads import zipf_offsets

    d, v, s, di, vi, si, T = host_inputs(name)
    B, N, V, H, r = d.B, d.N, d.V, d.H, d.r
    M = B * N
    # device-resident weights; the per-step inputs and the results the host reads back live in
    # one input and one output arena (one host<->device copy each way in the end-to-end leg)
    W = di["lm_head"].to(dev)
    w1 = di["w1"].to(dev)
    w2 = di["w2"].to(dev)
    h_in = {"X": di["hidden"], "anchor": torch.from_numpy(di["anchor"]), "temp": torch.from_numpy(T),
            "p_t": torch.from_numpy(vi["p_t"]), "p_d": torch.from_numpy(vi["p_d"]), "sps": torch.from_numpy(si["sps"])}
    in_specs = [(k, tuple(t.shape), t.dtype) for k, t in h_in.items()]
    out_specs = [("tok", (B, N), torch.int32), ("out", (B, N + 1), torch.int32), ("nacc", (B,), torch.int32),
                 ("K_out", (1,), torch.int32), ("lens", (B,), torch.int32), ("sel", (B * N,), torch.int32),
                 ("surv", (B, N), torch.float32), ("conf", (B, N), torch.float32)]
    d_in, d_out = Arena(in_specs, device=dev), Arena(out_specs, device=dev)
    for k, t in h_in.items():
        d_in.view(k).copy_(t)
    in_names = ("X", "anchor", "temp", "p_t", "p_d", "sps")
    step_inputs = tuple(d_in.view(k) for k in in_names)
    X, anchor, temp, p_t, p_d, sps = step_inputs
    tok, out, nacc, K_out, lens, sel, surv, conf = (d_out.view(k) for k in ("tok", "out", "nacc", "K_out", "lens", "sel",
                                                                            "surv", "conf"))
    # the calibrated confidence head's weights (synthetic): w_h ~ N(0, 1/H), w_e ~ N(0, 1/r), tau per position
    w_h, w_e, beta, tau = head_weights(d)
    w_h, w_e, tau = (torch.from_numpy(x).to(dev) for x in (w_h, w_e, tau))
    L = torch.empty(M, V, dtype=torch.float32, device=dev)
    ws_g = ds.Workspace(ds.OP_DRAFT_LOGITS, device=dev)
    ws_m = ds.Workspace(ds.OP_MARKOV_SAMPLE, B, N, V, r, device=dev)
    ws_v = ds.Workspace(ds.OP_VERIFY, B, N, V, device=dev)
    ws_s = ds.Workspace(ds.OP_SCHEDULE, B, N, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_sink = torch.empty((), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def flush_l2(k):
        # Write 512 MB (every L2 line replaced), then read back half of it: the read evicts
        # the dirty lines the write left behind, so their write-back happens here rather
        # than inside the next timed step.  The step starts with a cold, clean L2.
        flush.fill_(float(k))
        torch.sum(flush[: flush.numel() // 2], dim=0, out=flush_sink)

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]

    # The batched-draft workload defines its Markov-step logits as the base logits plus a
    # per-row Zipf(1.1) rank offset (peaked rows, as real LM logits are).  The offset is not
    # part of the method: it is drawn on the host (the same rows the oracle leg uses), added to
    # the GEMM output once before timing, and the sampler reads that buffer; both kernels still
    # do their full work every step.
    L_markov = L
    zipf_host = None
    if d.zipf > 0:
        zipf_host = zipf_offsets(d)
        ds.dspark_draft_logits(X, W, logits=L, workspace=ws_g)
        L_markov = torch.from_numpy(zipf_host).to(dev)
        L_markov += L
        torch.cuda.synchronize()

    # each replica serves its own requests: independent noise streams per rank
    seed_draft, seed_verify = replica_seed(0, rank), replica_seed(2, rank)

    # Verification reads the draft tokens and scheduling the head's confidences: neither needs
    # the other, so the step runs them on two streams (fork after the sampler, join at the end).
    # The eager pass that times each kernel runs them one after the other.
    sched_stream = torch.cuda.Stream(dev)

    def step(k=None, inp=None):
        # inp: (hidden, anchor, temperature, p_t, p_d, sps) views of another input arena
        X, anchor, temp, p_t, p_d, sps = inp if inp is not None else step_inputs
        e = ev[k] if k is not None else None
        cur = torch.cuda.current_stream()
        if e: e[0].record(stream)
        with _nvtx("dspark_draft_logits"):
            ds.dspark_draft_logits(X, W, logits=L, workspace=ws_g)
        if e: e[1].record(stream)
        with _nvtx("dspark_markov_sample_conf"):
            ds.dspark_markov_sample_conf(L_markov.view(B, N, V), anchor, w1, w2, temp, seed_draft, 0, X, w_h, w_e, beta,
                                         tau, draft_tokens=tok, conf=conf, workspace=ws_m)
        if e: e[2].record(stream)
        if e is None:
            sched_stream.wait_stream(cur)
            with torch.cuda.stream(sched_stream), _nvtx("dspark_schedule"):
                ds.dspark_schedule(conf, sps, -1, survival=surv, K_out=K_out, lengths=lens, selected=sel,
                                   workspace=ws_s)
        with _nvtx("dspark_verify"):
            ds.dspark_verify(p_t, p_d, tok, None, seed_verify, 0, out_tokens=out, num_accepted=nacc, workspace=ws_v)
        if e: e[3].record(stream)
        if e is None:
            cur.wait_stream(sched_stream)
        else:
            with _nvtx("dspark_schedule"):
                ds.dspark_schedule(conf, sps, -1, survival=surv, K_out=K_out, lengths=lens, selected=sel,
                                   workspace=ws_s)
            e[4].record(stream)

    for _ in range(args.warmup):
        flush_l2(1)
        step()
    torch.cuda.synchronize()
    for wsx in (ws_g, ws_m, ws_v, ws_s):
        st, bits = ds.dspark_read_status(wsx)
        if st not in (0,):
            raise RuntimeError(f"device status {st} bits {bits:#x} after warm-up")

    # The step is replayed as one CUDA graph (all buffers at fixed addresses, as a serving
    # engine runs its draft step); an eager pass with events between the calls gives the
    # per-kernel times used for the roofline.
    graph = None
    if not args.no_graph:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            step()
        for _ in range(args.warmup):
            flush_l2(1)
            graph.replay()
        torch.cuda.synchronize()
    g0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    g1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]

    # ---------------- timed region (device-resident inputs) ----------------
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        time.sleep(0.5)                           # let the sampler start before the timed region
        wall0 = time.perf_counter()
        for k in range(args.steps):
            flush_l2(k)                           # L2 flush between timed steps (not timed)
            if graph is not None:
                g0[k].record(stream)
                graph.replay()
                g1[k].record(stream)
            else:
                step(k)
        torch.cuda.synchronize()
        wall1 = time.perf_counter()
        wall = wall1 - wall0
        clk.mark(wall0, wall1)
        time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    if graph is not None:
        # per-kernel times: the same K steps run eagerly with events between the calls
        for k in range(args.steps):
            flush_l2(k)
            step(k)
        torch.cuda.synchronize()
    per = np.array([[ev[k][j].elapsed_time(ev[k][j + 1]) for j in range(4)] for k in range(args.steps)])
    kernel_ms = per.mean(axis=0)                  # draft_logits, markov, verify, schedule
    if graph is not None:
        step_ms = float(np.mean([a.elapsed_time(b) for a, b in zip(g0, g1)]))
    else:
        step_ms = float(per.sum(axis=1).mean())
    step_ms = max_over_ranks(step_ms, dist, dev)
    value = job_throughput(M, world, step_ms)

    # ---------------- roofline of the dominant kernel and of the sampler ----------------
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except OSError:
        pass
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    bf16_peak = float(peaks.get("bf16_tflops", 1900.0))
    peak_src = "measured" if peaks else "fallback"
    esize = 2 if d.dtype == "bf16" else 4
    gemm_bytes = (V * H + M * H) * esize + M * V * 4
    gemm_flops = 2.0 * M * H * V
    markov_bytes = M * V * 4 + V * r * esize + B * N * r * esize
    t_gemm = kernel_ms[0] / 1e3
    gemm_bound = "hbm" if gemm_bytes / (hbm_peak * 1e9) >= gemm_flops / (bf16_peak * 1e12) else "tensor"
    if gemm_bound == "hbm":
        ach = gemm_bytes / t_gemm / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": hbm_peak, "unit": "GB/s", "frac": ach / hbm_peak,
                "algorithmic_bytes_per_launch": gemm_bytes}
    else:
        ach = gemm_flops / t_gemm / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": bf16_peak, "unit": "TFLOP/s", "frac": ach / bf16_peak,
                "algorithmic_flops_per_launch": gemm_flops}
    roof["kernel"] = "dspark_draft_logits"
    roof["peak_source"] = peak_src
    tr = GEMM_TRAFFIC.get(name)
    roof["traffic"] = tr["bytes"] if tr is not None and tr["src_digest"] == gemm_source_digest() else None
    if roof["traffic"] is not None:
        roof["traffic_source"] = ("dram__bytes_read.sum + dram__bytes_write.sum of one ncu capture of "
                                  f"dspark_draft_logits on {name}")
    markov_roof = {"bound": "hbm", "algorithmic_bytes": markov_bytes,
                   "achieved": markov_bytes / (kernel_ms[1] / 1e3) / 1e9, "peak": hbm_peak,
                   "unit": "GB/s", "frac": markov_bytes / (kernel_ms[1] / 1e3) / 1e9 / hbm_peak,
                   "peak_source": peak_src}

    res = {
        "value": value, "ms_per_step": step_ms, "dtype": d.dtype,
        "config": {"workload": f"{d.name}: B={B} N={N} H={H} V={V} r={r} {d.dtype} "
                               f"T={WORKLOAD_TEMPERATURE[name]}, verify gamma={N}, "
                               f"schedule over B*N={M} candidates",
                   "global_batch_requests": B * world, "draft_tokens_per_step": M * world,
                   "parallelism": f"replicas x{world} (requests sharded, no collective)",
                   "l2": "flushed between timed steps: 512 MB write, then a 256 MB read-back that evicts the dirty lines",
                   "markov_input": ("base logits + per-row Zipf(1.1) rank offset (seeded host draw), offset "
                                    "applied once before timing" if d.zipf > 0 else "this step's base logits")},
        "kernel_ms": {"draft_logits": kernel_ms[0], "markov_sample": kernel_ms[1],
                      "verify": kernel_ms[2], "schedule": kernel_ms[3]},
        "roofline": roof,
        "markov_roofline": markov_roof,
        # per step: GEMM, Markov sampler with the confidence head and verify, each after its
        # workspace-clear kernel, then the scheduler (which clears its own status word)
        "gpu_launches": 7 * args.steps,
        "step_launch": ("one CUDA graph replay per step (verify and schedule on two streams after the sampler)"
                        if graph is not None else "four eager calls per step"),
        "kernel_ms_note": "per-kernel CUDA-event times from an eager pass over the same K steps",
        "clocks": clk.summary(),
        "wall_s_timed_region": wall,
    }
    if not full:
        return res

    # the step's outputs, read once for the oracle leg and the acceptance figures
    gpu_step = {"tok": tok.cpu().numpy(), "out": out.cpu().numpy(), "nacc": nacc.cpu().numpy(),
                "K": int(K_out.item()), "lens": lens.cpu().numpy(), "sel": sel.cpu().numpy(),
                "surv": surv.cpu().numpy(), "conf": conf.cpu().numpy()}
    tested = gpu_step["nacc"] + (gpu_step["nacc"] < N)
    res["step_verify"] = {"accepted_mean": float(gpu_step["nacc"].mean()),
                          "acceptance_rate": float(gpu_step["nacc"].sum() / max(1, tested.sum())),
                          "note": "empirical, over the step's requests: accepted tokens / tested positions "
                                  "(Markov draft tokens against the verify workload's p_t, p_d)"}

    # ---------------- end to end through host buffers ----------------
    e2e = None
    if not args.skip_e2e:
        # The step's inputs sit in one pinned host arena laid out like the device one and are
        # copied whole every step; the results are read back whole after every step.  Two device
        # input arenas: step k+1's inputs cross on a copy stream while step k runs from the other
        # arena (an event keeps a copy out of an arena until the step reading it is done).  The
        # timed region runs from the first step's copy to the last step's read-back; every
        # step's inputs (1.29 GB on the batched draft) are larger than L2, so no flush is added.
        hin, hout = Arena(in_specs, pin=True), Arena(out_specs, pin=True)
        for k, t in h_in.items():
            hin.view(k).copy_(t)
        h2d, d2h = hin.nbytes, hout.nbytes
        d_in2 = Arena(in_specs, device=dev)
        arenas = (d_in, d_in2)
        views = tuple(tuple(a.view(k) for k in in_names) for a in arenas)
        copy_stream = torch.cuda.Stream(dev)
        copied = [torch.cuda.Event() for _ in arenas]
        consumed = [torch.cuda.Event() for _ in arenas]

        def copy_in(j):
            copy_stream.wait_event(consumed[j])
            with torch.cuda.stream(copy_stream):
                arenas[j].buf.copy_(hin.buf, non_blocking=True)
            copied[j].record(copy_stream)

        def run(n):
            torch.cuda.synchronize()
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(copy_stream)
            copy_in(0)
            for k in range(n):
                j = k % 2
                if k + 1 < n:
                    copy_in(1 - j)
                stream.wait_event(copied[j])
                step(inp=views[j])
                hout.buf.copy_(d_out.buf, non_blocking=True)
                consumed[j].record(stream)
            t1.record(stream)
            torch.cuda.synchronize()
            return t0.elapsed_time(t1) / n

        run(args.warmup)
        e2e_ms = max_over_ranks(run(args.steps), dist, dev)
        e2e = {"value": job_throughput(M, world, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms,
               "note": "every step copies its inputs from pinned host memory and reads its results back; "
                       "step k+1's copy overlaps step k on a second stream (two device input arenas)"}
    res["e2e"] = e2e

    # ---------------- the library's other entry points, timed on their own ----------------
    # greedy verification of the step's draft tokens against the same target rows (all rows
    # k <= gamma are read)
    ws_g2 = ds.Workspace(ds.OP_VERIFY_GREEDY, B, N, device=dev)
    g_out = torch.empty(B, N + 1, dtype=torch.int32, device=dev)
    g_nacc = torch.empty(B, dtype=torch.int32, device=dev)
    greedy_ms = _timed_calls(lambda: ds.dspark_verify_greedy(p_t, tok, None, out_tokens=g_out, num_accepted=g_nacc,
                                                             workspace=ws_g2), flush_l2, stream)
    # the calibrated confidence head as its own launch (the step evaluates it inside the sampler)
    ws_c = ds.Workspace(ds.OP_CONFIDENCE, B, N, V, r, device=dev)
    conf_out = torch.empty(B, N, dtype=torch.float32, device=dev)
    conf_ms = _timed_calls(lambda: ds.dspark_confidence(X, w1, anchor, tok, w_h, w_e, beta, tau, conf=conf_out,
                                                        workspace=ws_c), flush_l2, stream)
    conf_bytes = M * H * X.element_size() + M * r * w1.element_size() + (H + r + N) * 4 + M * 4
    # the sampler on an EAGLE-3-sized reduced draft vocabulary (first 32000 entries of the step's
    # logits and Markov head, ids mapped into the target vocabulary through an index table)
    Vd = min(32000, V)
    L_red = L_markov.view(B, N, V)[:, :, :Vd].contiguous()
    w1_red, w2_red = w1[:Vd].contiguous(), w2[:Vd].contiguous()
    d2t = torch.from_numpy(np.sort(np.random.default_rng(d.data_seed + 8).choice(V, Vd, replace=False))
                           .astype(np.int32)).to(dev)
    ws_r = ds.Workspace(ds.OP_MARKOV_SAMPLE, B, N, Vd, r, device=dev)
    tok_red = torch.empty(B, N, dtype=torch.int32, device=dev)
    red_args = (L_red, anchor % Vd, w1_red, w2_red, temp, seed_draft, 0, d2t, ds.D2T_INDEX, V)
    red_ms = _timed_calls(lambda: ds.dspark_markov_sample_reduced(*red_args, draft_tokens=tok_red, workspace=ws_r),
                          flush_l2, stream)
    del L_red
    # verification straight from logits (the draft distribution never written): target logits
    # log p_t of the step's target rows, the step's draft base logits, tokens and sampler lse
    lse_d = torch.empty(B, N, dtype=torch.float32, device=dev)
    ws_m2 = ds.Workspace(ds.OP_MARKOV_SAMPLE, B, N, V, r, device=dev)
    tok_l = torch.empty(B, N, dtype=torch.int32, device=dev)
    ds.dspark_markov_sample(L_markov.view(B, N, V), anchor, w1, w2, temp, seed_draft, 0, draft_tokens=tok_l,
                            lse=lse_d, workspace=ws_m2)
    # target logits that follow the draft: the draft's base logit rows (the last one again for the
    # bonus position) plus N(0, sigma_b^2) noise, sigma_b in {0.3, 1, 3} per request
    gen_t = torch.Generator(device=dev)
    gen_t.manual_seed(d.data_seed + 9)
    sig = torch.tensor([0.3, 1.0, 3.0], device=dev)[torch.randint(0, 3, (B,), generator=gen_t, device=dev)]
    Lm = L_markov.view(B, N, V)
    t_logits = torch.cat([Lm, Lm[:, -1:]], dim=1) + sig[:, None, None] * torch.randn(
        B, N + 1, V, generator=gen_t, device=dev)
    del Lm
    T_t = torch.ones(B, dtype=torch.float32, device=dev)
    ws_l = ds.Workspace(ds.OP_VERIFY_LOGITS, B, N, V, r, device=dev)
    l_out = torch.empty(B, N + 1, dtype=torch.int32, device=dev)
    l_nacc = torch.empty(B, dtype=torch.int32, device=dev)
    vl_args = (t_logits, T_t, L_markov.view(B, N, V), anchor, w1, w2, temp, lse_d, tok_l, None, seed_verify, 0)
    vlog_ms = _timed_calls(lambda: ds.dspark_verify_logits(*vl_args, out_tokens=l_out, num_accepted=l_nacc,
                                                           workspace=ws_l), flush_l2, stream)
    # bytes a request needs: its target rows k <= k* once for the normalisers (k* = the number
    # accepted, N if none was rejected) and row k* once more for the draw; the draft's base logits
    # and Markov rows are read only at the few candidate entries
    vlog_rows = int((l_nacc.long() + 2).sum().item())
    vlog_bytes = vlog_rows * V * 4
    # verification with the draft's own Gumbel noise on the same target logits (the draft's
    # temperature for the target, the sampler's seed and offset); all rows k <= gamma are read
    ws_gu = ds.Workspace(ds.OP_VERIFY_GUMBEL, B, N, device=dev)
    gu_out = torch.empty(B, N + 1, dtype=torch.int32, device=dev)
    gu_nacc = torch.empty(B, dtype=torch.int32, device=dev)
    gu_args = (t_logits, temp, tok_l, None, seed_draft, 0)
    gumbel_ms = _timed_calls(lambda: ds.dspark_verify_gumbel(*gu_args, out_tokens=gu_out, num_accepted=gu_nacc,
                                                             workspace=ws_gu), flush_l2, stream)
    gumbel_bytes = B * (N + 1) * V * 4
    del ws_l, ws_m2, t_logits
    # confidence-scheduled admission under load: B=1024 requests x N=16 candidates, SPS over batch
    # sizes 1..16384, K chosen (its own launches, outside the step); cold = L2 flushed before each
    # call, warm = 20 calls back to back
    sc = SCHEDULE_CONFIGS["schedule"]
    sci = schedule_inputs(sc)
    c_sc = torch.from_numpy(sci["cond_accept"]).to(dev)
    sps_sc = torch.from_numpy(sci["sps"]).to(dev)
    ws_sc = ds.Workspace(ds.OP_SCHEDULE, sc.B, sc.N, device=dev)
    sc_out = (torch.empty(sc.B * sc.N, dtype=torch.float32, device=dev), torch.empty(1, dtype=torch.int32, device=dev),
              torch.empty(sc.B, dtype=torch.int32, device=dev), torch.empty(sc.B * sc.N, dtype=torch.int32, device=dev))

    def sched_call():
        ds.dspark_schedule(c_sc, sps_sc, -1, survival=sc_out[0], K_out=sc_out[1], lengths=sc_out[2],
                           selected=sc_out[3], workspace=ws_sc)

    sched_cold_ms = _timed_calls(sched_call, flush_l2, stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(20):
        sched_call()
    e1.record(stream)
    torch.cuda.synchronize()
    sched_warm_ms = e0.elapsed_time(e1) / 20

    def hbm_entry(ms, nbytes, note, **extra):
        e = {"ms": ms, "bound": "hbm", "algorithmic_bytes": nbytes, "achieved": nbytes / (ms / 1e3) / 1e9,
             "peak": hbm_peak, "unit": "GB/s", "frac": nbytes / (ms / 1e3) / 1e9 / hbm_peak, "note": note}
        e.update(extra)
        return e

    res["markov_sample_reduced_vocab"] = {"ms": red_ms, "draft_vocab": Vd, "target_vocab": V,
                                          "note": "median of 20 launches, L2 flushed, outside the step"}
    res["confidence_standalone"] = hbm_entry(conf_ms, conf_bytes, "dspark_confidence as its own launch: median of 20 "
                                             "launches, L2 flushed, outside the step (the step evaluates the head "
                                             "inside dspark_markov_sample_conf)")
    res["verify_logits"] = hbm_entry(vlog_ms, vlog_bytes,
                                     "median of 20 calls (2 kernels), L2 flushed, outside the step; bytes = "
                                     "target rows k <= k* plus row k* again, from the measured k*",
                                     accepted_mean=float(l_nacc.float().mean().item()),
                                     target="the draft's base-logit rows + N(0, s^2), s in {0.3, 1, 3} per request")
    res["verify_gumbel"] = hbm_entry(gumbel_ms, gumbel_bytes,
                                     "median of 20 launches, L2 flushed, outside the step; target logits as for "
                                     "verify_logits, the draft's temperature and noise",
                                     accepted_mean=float(gu_nacc.float().mean().item()))
    res["verify_greedy"] = hbm_entry(greedy_ms, B * (N + 1) * V * 4,
                                     "median of 20 launches, L2 flushed, outside the step")
    res["schedule_b1024_n16"] = {"ms": sched_cold_ms, "warm_ms": sched_warm_ms, "candidates": sc.B * sc.N,
                                 "K": int(sc_out[1].item()),
                                 "note": "dspark_schedule per call (one kernel on a cluster of 16 blocks; it clears "
                                         "its own status word): ms = median of 20 calls with L2 flushed before "
                                         "each, warm_ms = mean of 20 calls back to back"}
    res["_oracle_inputs"] = (d, v, s, di, vi, si, T, None if zipf_host is None else zipf_host.__getitem__,
                             gpu_step)
    return res


def run_gpu(args):
    import torch
    import draft_sampling_verification_tcgen05_gb300 as ds
    from draft_sampling_verification_tcgen05_gb300 import _build
    from draft_sampling_verification_tcgen05_gb300.replicas import rank_info

    ri = rank_info()
    rank, world, local = ri.rank, ri.world, ri.local_rank
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or world == 1:
        _build.build()
    if dist is not None:
        dist.barrier()
    ds.lib()

    main_res = measure(args.workload, args, dev, dist, world, rank, full=True)
    oracle_inputs = main_res.pop("_oracle_inputs")
    secondary = None
    if args.secondary != "none" and args.secondary != args.workload:
        torch.cuda.empty_cache()
        sec = measure(args.secondary, args, dev, dist, world, rank, full=False)
        secondary = {"workload": sec["config"]["workload"], "value": sec["value"], "unit": UNIT,
                     "ms_per_step": sec["ms_per_step"], "kernel_ms": sec["kernel_ms"],
                     "roofline": sec["roofline"], "markov_roofline": sec["markov_roofline"],
                     "clocks": sec["clocks"], "gpu_launches": sec["gpu_launches"],
                     "note": "same step, timing and L2 flush as the headline workload"}

    if dist is not None and rank != 0:
        dist.barrier()
        dist.destroy_process_group()
        return

    res = {"metric": METRIC, "value": main_res.pop("value"), "unit": UNIT, "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": main_res.pop("ms_per_step"), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": main_res.pop("dtype"), "data": "synthetic"}
    res.update(main_res)
    if secondary is not None:
        res["gpu_launches"] += secondary["gpu_launches"]
        res["secondary"] = secondary
    if not args.skip_cpu_baseline and rank == 0:
        res["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_seconds, oracle_inputs)
    print(json.dumps(res))
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# CPU oracle (baseline leg and reference arm)
# ---------------------------------------------------------------------------
def _blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def oracle_step(inputs, req, gpu=None, parity=None):
    """The whole hot path on the CPU oracle for the requests `req` of one batch.

    With `gpu` (the GPU step's outputs), the sampler runs teacher-forced on the GPU's draft
    tokens and verification takes the GPU's tokens, so that `parity` can count how the two
    agree (the oracle's work per step is the same either way)."""
    import oracle
    d, v, s, di, vi, si, T, zipf_of = inputs[:8]
    rows = (req[:, None] * d.N + np.arange(d.N)[None, :]).reshape(-1)
    Lr = oracle.draft_logits(di["hidden_f32"][rows], di["lm_head_f32"])
    if zipf_of is not None:
        Lr = Lr + zipf_of(rows)
    Lr = Lr.reshape(len(req), d.N, d.V)
    forced = None if gpu is None else gpu["tok"][req].astype(np.int64)
    tok, gap, _ = oracle.markov_sample(Lr, di["anchor"][req], di["w1_f32"], di["w2_f32"], T[req], 0, 0,
                                       req_ids=req, forced_tokens=forced)
    x = tok if gpu is None else forced
    w_h, w_e, beta, tau = head_weights(d)
    c = oracle.confidence(di["hidden_f32"][rows], di["w1_f32"], di["anchor"][req], x, w_h, w_e, beta, tau)
    out, nacc, _, _ = oracle.verify(vi["p_t"][req], vi["p_d"][req], x, None, 2, 0, req_ids=req)
    oracle.schedule(c.astype(np.float32), si["sps"][: len(req) * d.N], -1)
    if parity is not None and gpu is not None:
        diff = tok != forced
        parity["markov_compared"] += int(tok.size)
        parity["markov_near_tie"] += int((diff & (gap < 5e-2)).sum())
        parity["markov_mismatch"] += int((diff & (gap >= 5e-2)).sum())
        parity["verify_compared"] += len(req)
        parity["verify_mismatch"] += int(np.sum(np.any(out != gpu["out"][req], axis=1) | (nacc != gpu["nacc"][req])))
        parity["confidence_max_abs_diff"] = max(parity.get("confidence_max_abs_diff", 0.0),
                                                float(np.abs(c - gpu["conf"][req]).max()))
    return len(req) * d.N


ONE_THREAD_ENV = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS")


def oracle_single_thread(name):
    """One request of the workload through the oracle in a child process whose BLAS runs on one
    thread (numpy's own array work is single-threaded already)."""
    env = dict(os.environ, **{k: "1" for k in ONE_THREAD_ENV})
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-one-request", "--workload", name],
                       env=env, capture_output=True, text=True, timeout=600)
    if r.returncode != 0:
        return {"unavailable": (r.stderr.strip().splitlines() or ["child failed"])[-1]}
    line = json.loads(r.stdout.strip().splitlines()[-1])
    return {"value": line["tokens"] / line["seconds"], "unit": UNIT, "cores": 1,
            "sample": f"1 request: {line['tokens']} draft tokens in {line['seconds']:.1f} s (BLAS on 1 thread)"}


def run_oracle_one_request(args):
    from workloads import zipf_offsets
    d, v, s = step_configs(args.workload)
    di = draft_inputs(d)
    vi = verify_inputs(v, B=1)
    si = schedule_inputs(s, B=1)
    T = np.full(d.B, WORKLOAD_TEMPERATURE[args.workload], np.float32)
    zipf_of = (lambda rows: zipf_offsets(d, rows)) if d.zipf > 0 else None
    t0 = time.perf_counter()
    n = oracle_step((d, v, s, di, vi, si, T, zipf_of), np.array([0]))
    print(json.dumps({"tokens": n, "seconds": time.perf_counter() - t0}))


def cpu_baseline(name, budget_s, inputs):
    """The oracle, as it stands, on a bounded sample of the workload's requests: all BLAS threads
    (about budget_s seconds), then one request on one thread.  The sampled requests are compared
    with the GPU step's outputs (teacher-forced sampler, verification on the GPU's tokens), and
    the full scheduling pool is scheduled by the oracle and compared bit for bit."""
    import oracle
    d = inputs[0]
    gpu = inputs[8]
    si = inputs[5]
    parity = {"markov_compared": 0, "markov_near_tie": 0, "markov_mismatch": 0,
              "verify_compared": 0, "verify_mismatch": 0}
    t0 = time.perf_counter()
    tokens = 0
    b = 0
    stride = max(1, d.B // 8 + 1) if d.B > 1 else 1
    while True:
        req = np.array([(b * stride) % d.B])
        tokens += oracle_step(inputs, req, gpu, parity)
        b += 1
        if time.perf_counter() - t0 >= budget_s or b >= d.B:
            break
    el = time.perf_counter() - t0
    one = oracle_single_thread(name)
    rs = oracle.schedule(gpu["conf"], si["sps"], -1)          # the head's float32 confidences, as the GPU's input
    sched_ok = (rs["K"] == gpu["K"] and np.array_equal(rs["lengths"], gpu["lens"])
                and np.array_equal(rs["selected"], gpu["sel"]) and np.array_equal(rs["survival"], gpu["surv"]))
    parity["schedule_pool"] = int(si["cond_accept"].size)
    parity["schedule_bit_exact"] = bool(sched_ok)
    parity["note"] = ("sampled requests: the oracle's tokens teacher-forced on the GPU step's tokens (a token "
                      "may differ only at an oracle top-2 gap < 5e-2: near_tie; mismatch counts the rest), "
                      "the confidence head on the GPU's tokens (tolerance 2e-5), verification of the GPU's "
                      "tokens compared bit for bit per request; the whole scheduling pool (the head's float32 "
                      "confidences) compared bit for bit")
    return {"value": tokens / el, "unit": UNIT, "cores": _blas_threads(), "kind": "oracle",
            "sample": f"{b} request(s) of {d.name} through the whole path on the CPU oracle "
                      f"(fp64 numpy): {tokens} draft tokens in {el:.1f} s",
            "single_thread": one,
            "parity": parity}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    d, v, s, di, vi, si, T = host_inputs(args.workload)
    zipf_of = None
    if d.zipf > 0:
        from workloads import zipf_offsets
        zipf_host = zipf_offsets(d)
        zipf_of = zipf_host.__getitem__
    inputs = (d, v, s, di, vi, si, T, zipf_of)
    per_step_budget = max(1.0, args.cpu_seconds / max(1, args.steps))
    for _ in range(args.warmup):
        oracle_step(inputs, np.array([0]))
    times, toks = [], 0
    for k in range(args.steps):
        t0 = time.perf_counter()
        n = 0
        b = k
        while True:
            n += oracle_step(inputs, np.array([b % d.B]))
            b += args.steps
            if time.perf_counter() - t0 >= per_step_budget or n >= d.B * d.N:
                break
        times.append(time.perf_counter() - t0)
        toks += n
    value = toks / sum(times)
    res = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * float(np.mean(times)),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic",
           "config": {"workload": f"{d.name}: B={d.B} N={d.N} H={d.H} V={d.V} r={d.r} {d.dtype}",
                      "note": "CPU oracle, each step a bounded sample of requests of the workload"},
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": _blas_threads(), "kind": "oracle",
                            "sample": f"{toks} draft tokens over {args.steps} steps"},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res))


def main():
    args = parse()
    if args.oracle_one_request:
        run_oracle_one_request(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
