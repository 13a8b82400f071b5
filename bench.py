"""Benchmark of the KDA bounded-gate prefill (and verify) on GB300.

One step = one kda_chunk_prefill call over the 8 x 2048-token, H=16, d=128
workload (initial states gathered from a 64-slot pool, dense final states),
inputs resident in HBM.  The call is two launches: the intra-chunk kernel over
every (chunk, head) and the state pass over every (sequence, head); the
roofline line covers the whole call (its algorithmic bytes over its
CUDA-event time), the per-kernel split is in profiles/.  Also timed: the same call end to end with host
buffers (pinned H2D of the step's inputs + D2H of its outputs inside the
timed region), the verify call on 64 requests x 8, 4 and 1 tokens and the
accept/commit after it (each captured in a CUDA graph and replayed, the way a
serving step runs them), one speculative-decoding step (a 4 x 2048-token
prefill segment beside 64 verify requests x 4 tokens, every output row stored
by index into the layer output), the other prefill workloads (1 x 256 at H=2,
4 x 8192, and 16384 + 16 varlen sequences with its long sequence also timed
alone) as their own calls -- the long ones take the split state-pass schedule
by default and are also timed on the plain two-kernel schedule and on the
fused kernel -- and the fp64 CPU oracle on each workload (bounded
samples where the whole would take long).  Per-call times are CUDA events on
the launching stream and the reported per-layer figures are their median; SM
clocks are sampled through NVML inside the timed region.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
N > 1 runs under torchrun, one replica per GPU (weak scaling, no collective on
the data path; a barrier and a max over ranks bracket the timing).
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA prefill tokens/s per layer (H=16,d=128) and % roofline; verify µs/layer"
WORKLOAD = "prefill_2048x8_h16"
PAGES_FLASHKDA_US = 49.0  # vLLM PR #55737 (GB300, T=2048x8, per layer): context, another kernel
L2_BYTES = 129e6
TOKEN_HEAD_BYTES = 4 * 256 + 2 + 256  # q, k, v, g + beta + out (bf16)
STATE_BYTES = 128 * 128 * 4


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def prefill_algorithmic_bytes(inp):
    T, H = inp.total_tokens, inp.H
    states = inp.num_seqs * H * STATE_BYTES * ((1 if inp.load_initial else 0) + 1)
    return T * H * TOKEN_HEAD_BYTES + states


def verify_algorithmic_bytes(inp):
    BT, H = inp.B * inp.T, inp.H
    return BT * H * TOKEN_HEAD_BYTES + inp.B * H * STATE_BYTES * (1 + inp.T)


# the gated RMSNorm of an output row and head: the bf16 gate row read and the fp32 rstd written
NORM_BYTES_PER_ROW = 256 + 4
# one short-convolution window of a (sequence or step, head): 3 raw inputs of q, k and v, bf16
CONV_WINDOW_BYTES = 3 * 3 * 128 * 2


def spec_step_algorithmic_bytes(inp):
    """Both segments' bytes (prefill: initial and final state per sequence and head) plus the int32 row index of
    every token."""
    p, v = inp.prefill, inp.verify
    return (prefill_algorithmic_bytes(p) + verify_algorithmic_bytes(v) +
            4 * (p.total_tokens + v.B * v.T))


# sources that decide each kernel's code (a traffic record is valid while they are unchanged)
KERNEL_SOURCES = {
    "prefill": ("kda_chunk_intra.cu", "kda_chunk_chain.cu", "kda_prefill.cu", "kda_prefill_block.h", "kda_sm100.cuh",
                "kda_common.cuh", "kda_internal.h"),
    "verify": ("kda_recurrent.cu", "kda_common.cuh", "kda_internal.h"),
    "prefill_fused": ("kda_prefill_fused.cu", "kda_prefill.cu", "kda_prefill_block.h", "kda_sm100.cuh", "kda_common.cuh",
                      "kda_internal.h"),
}


def source_digest(kind):
    csrc = os.path.join(ROOT, "kda_linear_attention_bounded_gb300", "csrc")
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kind]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kind):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", f"{kind}_traffic.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("source_digest") != source_digest(kind):
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class _Nvml:
    """NVML through ctypes (reads only): SM clock, its maximum and the active clock-event reasons."""

    # nvmlClocksEventReasons bits (nvml.h)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}
    CLOCK_SM = 1

    def __init__(self, uuid):
        import ctypes
        self.ct = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) != 0:
            raise OSError(f"no NVML device {uuid}")
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.lib = lib
        v = ctypes.c_uint(0)
        lib.nvmlDeviceGetMaxClockInfo(self.h, self.CLOCK_SM, ctypes.byref(v))
        self.max_mhz = float(v.value)

    def sample(self):
        ct = self.ct
        clk = ct.c_uint(0)
        rs = ct.c_ulonglong(0)
        if self.lib.nvmlDeviceGetClockInfo(self.h, self.CLOCK_SM, ct.byref(clk)) != 0:
            return None
        self.reasons_fn(self.h, ct.byref(rs))
        return float(clk.value), self.max_mhz, [n for bit, n in self.REASONS.items() if rs.value & bit]


class ClockSampler:
    """SM clock and throttle reasons sampled while running: through NVML every 0.5 ms (so that samples land
    inside even a few-millisecond timed region), else nvidia-smi every 50 ms."""

    FIELDS = "clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown," \
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown," \
             "clocks_event_reasons.sw_power_cap"
    SMI_NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device_index):
        self.device_index = device_index
        self.samples = []   # (time, sm_mhz, sm_max_mhz, [reasons])
        self.proc = None
        self.nvml = None
        self.running = False
        self.t0 = self.t1 = None
        self.source = None

    def start(self):
        try:
            import torch
            uuid = "GPU-" + str(torch.cuda.get_device_properties(self.device_index).uuid)
            self.nvml = _Nvml(uuid)
            self.source = "nvml, 0.5 ms"
        except Exception:
            self.nvml = None
        self.running = True
        if self.nvml is not None:
            threading.Thread(target=self._poll, daemon=True).start()
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(self.device_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi, 50 ms"
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _poll(self):
        while self.running:
            s = self.nvml.sample()
            if s is not None:
                self.samples.append((time.time(), *s))
            time.sleep(0.0005)

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                reasons = [self.SMI_NAMES[i] for i, v in enumerate(parts[3:7]) if v.lower() == "active"]
                self.samples.append((time.time(), float(parts[0]), float(parts[1]), reasons))
            except ValueError:
                continue

    def mark(self, which):
        if which == "begin":
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        self.running = False
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        time.sleep(0.01)
        rows = list(self.samples)
        inside = [r for r in rows if self.t0 and self.t1 and self.t0 <= r[0] <= self.t1]
        use = inside or rows
        if not use:
            return None
        reasons = sorted({n for r in use for n in r[3]})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use), "in_timed_region": bool(inside), "source": self.source}


def dist_setup(n_gpus):
    import torch
    import torch.distributed as dist

    if n_gpus > 1 or "RANK" in os.environ:
        rank = int(os.environ.get("RANK", 0))
        world = int(os.environ.get("WORLD_SIZE", 1))
        local = int(os.environ.get("LOCAL_RANK", 0))
        torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        return rank, world, local
    return 0, 1, 0


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device=None):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# reference arm: the fp64 CPU oracle, as it stands, on the host cores
# ---------------------------------------------------------------------------

def oracle_sample_rate(inp, seqs, tokens, nthreads):
    """Run the oracle on the first `seqs` sequences x all heads, the first `tokens` tokens of each (fewer where a
    sequence is shorter); return (token-rows processed, seconds)."""
    import numpy as np
    import oracle

    starts = inp.cu_seqlens[:seqs]
    lens = [min(tokens, int(inp.cu_seqlens[i + 1] - inp.cu_seqlens[i])) for i in range(seqs)]
    rows = np.concatenate([np.arange(s, s + n) for s, n in zip(starts, lens)])
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    S0 = inp.initial_states()[:seqs] if inp.load_initial else None
    t0 = time.perf_counter()
    oracle.run(inp.q[rows], inp.k[rows], inp.v[rows], inp.g[rows], inp.beta[rows], inp.A_log, inp.dt_bias,
               inp.lower_bound, inp.scale, cu, S0=S0, nthreads=nthreads)
    return int(cu[-1]), time.perf_counter() - t0


def cpu_baseline(inp, budget_s=30.0):
    """The oracle on the host cores: the whole workload (all sequences and heads), shortened per sequence only if
    a calibration run predicts more than `budget_s` seconds of wall time on those cores."""
    import oracle

    oracle.build()
    nthreads = oracle.default_threads()
    seqs = inp.num_seqs
    longest = int(max(inp.cu_seqlens[1:] - inp.cu_seqlens[:-1]))
    tok, dt = oracle_sample_rate(inp, seqs, 64, nthreads)  # calibration
    wall_s_per_token = dt / tok
    tokens = int(min(longest, max(64, budget_s / wall_s_per_token / seqs)))
    tok, dt = oracle_sample_rate(inp, seqs, tokens, nthreads)
    what = "the whole workload" if tokens >= longest else f"first {tokens} tokens of each sequence"
    return {"value": tok / dt, "unit": "tokens/s", "cores": nthreads, "kind": "oracle",
            "us_per_layer_equiv": dt * 1e6 * inp.total_tokens / tok,
            "sample": f"{what}: {seqs} sequences x all {inp.H} heads ({tok} tokens), fp64 token-by-token, "
                      f"{dt:.2f} s wall on {nthreads} threads (~{dt * nthreads:.0f} core-s)"}


def cpu_baseline_verify(inp):
    """The oracle on a verify workload (every request and head, every per-step state recorded)."""
    import oracle

    oracle.build()
    nthreads = oracle.default_threads()
    t0 = time.perf_counter()
    oracle.run_verify(inp, nthreads=nthreads)
    dt = time.perf_counter() - t0
    return {"value": dt * 1e6, "unit": "us/layer", "cores": nthreads, "kind": "oracle",
            "sample": f"the whole workload: {inp.B} requests x {inp.T} tokens x all {inp.H} heads with every "
                      f"per-step state, fp64 token-by-token, {dt:.2f} s wall on {nthreads} threads"}


def run_reference(args):
    rank = int(os.environ.get("RANK", 0))
    if rank != 0:
        return
    import oracle
    from kda_linear_attention_bounded_gb300 import inputs

    oracle.build()
    inp = inputs.prefill_2048x8()
    nthreads = oracle.default_threads()
    seqs = min(inp.num_seqs, max(1, nthreads // inp.H) or 1)
    tok, dt = oracle_sample_rate(inp, seqs, 64, nthreads)
    per_step_budget = 150.0 / max(1, args.steps + args.warmup)
    tokens = int(min(2048, max(16, per_step_budget * (tok / dt) / seqs)))
    for _ in range(args.warmup):
        oracle_sample_rate(inp, seqs, tokens, nthreads)
    total_tok = 0
    total_t = 0.0
    for _ in range(args.steps):
        t, d = oracle_sample_rate(inp, seqs, tokens, nthreads)
        total_tok += t
        total_t += d
    value = total_tok / total_t
    sample = f"per step {seqs} sequence(s) x all {inp.H} heads x first {tokens} tokens of {WORKLOAD}"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "H": inp.H, "d": 128, "tokens_per_step": total_tok // args.steps},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": nthreads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_gpu(args):
    import numpy as np
    import torch

    rank, world, local = dist_setup(args.gpus)
    device = torch.device("cuda", local)
    import kda_linear_attention_bounded_gb300 as kda
    from kda_linear_attention_bounded_gb300 import inputs
    from kda_linear_attention_bounded_gb300.device import DevicePrefill, DeviceSpecStep, DeviceVerify, bf16_dev, f32_dev

    kda.load()
    inp = inputs.prefill_2048x8()
    dev = DevicePrefill(inp, device=device)
    ws = dev.workspace(device)
    stream = torch.cuda.current_stream(device)
    H, T = inp.H, inp.total_tokens
    out = torch.empty((T, H, 128), dtype=torch.bfloat16, device=device)
    final = torch.empty((inp.num_seqs, H, 128, 128), dtype=torch.float32, device=device)

    def step():
        dev.run(out=out, final_state=final, workspace=ws, stream=stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(device)

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.2)
    switch = sys.getswitchinterval()
    sys.setswitchinterval(0.0002)   # lets the sampling thread run between the step launches
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(device)
    if sampler:
        sampler.mark("begin")
    t_wall = time.perf_counter()
    for i in range(args.steps):
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(device)
    barrier(world)
    wall = time.perf_counter() - t_wall
    if sampler:
        sampler.mark("end")
    sys.setswitchinterval(switch)
    per_launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    elapsed_ms = starts[0].elapsed_time(ends[-1])
    elapsed_ms = max_over_ranks(elapsed_ms, world, device)
    clocks = sampler.stop() if sampler else None
    assert kda.read_device_status(ws) == 0

    tokens_all = T * args.steps * world
    value = tokens_all / (elapsed_ms / 1e3)
    avg_launch_s = statistics.mean(per_launch_ms) / 1e3
    med_launch_s = statistics.median(per_launch_ms) / 1e3
    peak, peak_kind = measured_peaks()
    alg = prefill_algorithmic_bytes(inp)
    achieved = alg / med_launch_s / 1e9

    # ---- end to end through the C ABI with host buffers ----
    # Every step copies its inputs from pinned host memory, runs the call and copies its outputs back.  The
    # steps are pipelined the way a serving loop runs them: step i+1's host-to-device copies (own stream)
    # overlap step i's kernels, and step i's device-to-host copies (own stream) overlap step i+1's; device
    # buffers are double-buffered and ordered by events.
    host = {name: getattr(dev, name).cpu().pin_memory() for name in ("q", "k", "v", "g", "beta")}
    out_h = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    final_h = [torch.empty(final.shape, dtype=final.dtype).pin_memory() for _ in range(2)]
    bufs = [{name: torch.empty_like(getattr(dev, name)) for name in host} for _ in range(2)]
    outs = [torch.empty_like(out) for _ in range(2)]
    finals = [torch.empty_like(final) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h[0].numel() * out_h[0].element_size() + final_h[0].numel() * final_h[0].element_size()
    e2e_steps = max(3, min(args.steps, 100))
    s_h2d = torch.cuda.Stream(device)
    s_d2h = torch.cuda.Stream(device)
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("h2d", "comp", "d2h")}
    for k in ev:
        for e in ev[k]:
            e.record(stream)

    copy_ev = []   # per step: (H2D start, H2D end, D2H start, D2H end) on the copy streams

    def e2e_step(i):
        b = i & 1
        marks = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        with torch.cuda.stream(s_h2d):
            s_h2d.wait_event(ev["comp"][b])          # the call that last read buffer b has finished
            marks[0].record(s_h2d)
            for name, t in host.items():
                bufs[b][name].copy_(t, non_blocking=True)
            marks[1].record(s_h2d)
            ev["h2d"][b].record(s_h2d)
        stream.wait_event(ev["h2d"][b])
        stream.wait_event(ev["d2h"][b])              # output buffer b has been copied out
        kda.chunk_prefill(bufs[b]["q"], bufs[b]["k"], bufs[b]["v"], bufs[b]["g"], bufs[b]["beta"], dev.A_log,
                          dev.dt_bias, dev.cu, dev.cu_host, lower_bound=inp.lower_bound, scale=inp.scale,
                          state_pool=dev.pool, slot_ids=dev.slots, load_initial=True, out=outs[b],
                          final_state=finals[b], workspace=ws, stream=stream)
        ev["comp"][b].record(stream)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(ev["comp"][b])
            marks[2].record(s_d2h)
            out_h[b].copy_(outs[b], non_blocking=True)
            final_h[b].copy_(finals[b], non_blocking=True)
            marks[3].record(s_d2h)
            ev["d2h"][b].record(s_d2h)
        copy_ev.append(marks)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize(device)
    copy_ev.clear()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_h2d)
    for i in range(e2e_steps):
        e2e_step(i)
    s_h2d.wait_stream(s_d2h)
    e1.record(s_h2d)
    torch.cuda.synchronize(device)
    barrier(world)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, device)
    e2e_value = T * e2e_steps * world / (e2e_ms / 1e3)
    h2d_ms = statistics.median(m[0].elapsed_time(m[1]) for m in copy_ev)
    d2h_ms = statistics.median(m[2].elapsed_time(m[3]) for m in copy_ev)
    copy_ev.clear()
    # the results of the last step came back intact
    assert torch.equal(out_h[(e2e_steps - 1) & 1], outs[(e2e_steps - 1) & 1].cpu())
    del bufs, outs, finals

    # ---- verify (64 requests x 8, 4 and 1 tokens) and accept/commit, timed as CUDA-graph replays ----
    def graph_time_us(calls, steps):
        """Mean µs per call of ``calls`` (callables on the current stream) captured once
        in a CUDA graph and replayed; the calls rotate so each one sees cold L2."""
        side = torch.cuda.Stream(device)
        side.wait_stream(torch.cuda.current_stream(device))
        with torch.cuda.stream(side):
            for c in calls:
                c()
        torch.cuda.current_stream(device).wait_stream(side)
        torch.cuda.synchronize(device)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for c in calls:
                c()
        for _ in range(3):
            graph.replay()
        reps = max(3, math.ceil(steps / len(calls)))
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(device)
        g0.record()
        for _ in range(reps):
            graph.replay()
        g1.record()
        torch.cuda.synchronize(device)
        return g0.elapsed_time(g1) * 1e3 / (reps * len(calls)), reps * len(calls)

    def time_verify(vin):
        """One verify call per rotation set: disjoint slot sets and separate per-step buffers, as many as it
        takes for one rotation to move more than 3x the L2 (the pool rows and states are then read cold)."""
        vdev = DeviceVerify(vin, device=device)
        per_call = verify_algorithmic_bytes(vin)
        n_rot = min(vin.pool.shape[0] // vin.B, max(1, math.ceil(3 * L2_BYTES / per_call)))
        others = np.setdiff1d(np.arange(vin.pool.shape[0]), vin.slot_ids)
        others = np.random.default_rng(11).permutation(others)
        slot_sets = [vdev.slots] + [torch.from_numpy(others[r * vin.B:(r + 1) * vin.B].astype(np.int32)).to(device)
                                    for r in range(n_rot - 1)]
        vout = torch.empty((vin.B * vin.T, H, 128), dtype=torch.bfloat16, device=device)
        inters = [torch.empty((vin.B, vin.T, H, 128, 128), dtype=torch.float32, device=device) for _ in range(n_rot)]

        def call(r):
            return lambda: kda.recurrent_verify(vdev.q, vdev.k, vdev.v, vdev.g, vdev.beta, vdev.A_log, vdev.dt_bias,
                                                vdev.pool, slot_sets[r], vin.T, lower_bound=vin.lower_bound,
                                                scale=vin.scale, out=vout, intermediate_states=inters[r],
                                                workspace=ws)
        us, n = graph_time_us([call(r) for r in range(n_rot)], max(3, min(args.steps, 200)))
        achieved = per_call / (us * 1e-6) / 1e9
        rec = {"workload": vin.name, "T": vin.T, "us_per_layer": us, "calls_timed": n, "rotation_sets": n_rot,
               "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                            "frac": achieved / peak, "traffic": None, "algorithmic_bytes": per_call}}
        return rec, vdev, inters[0]

    vrec, vdev, inter = time_verify(inputs.verify_64x8())
    vrec["roofline"]["traffic"] = recorded_traffic("verify")
    vvariants = [time_verify(make())[0] for make in (inputs.verify_64x4, inputs.verify_64x1)]
    vin = vdev.inp

    # ---- accept/commit after verify: 1..8 accepted tokens per request ----
    n_acc = torch.from_numpy(np.random.default_rng(7).integers(1, vin.T + 1, size=vin.B).astype(np.int32)).to(device)
    c_us, c_steps = graph_time_us(
        [lambda: kda.commit_accepted(vdev.pool, vdev.slots, n_acc, inter, workspace=ws)], max(3, min(args.steps, 200)))
    c_bytes = 2 * vin.B * H * STATE_BYTES
    c_achieved = c_bytes / (c_us * 1e-6) / 1e9
    assert kda.read_device_status(ws) == 0

    del inter

    # ---- the same prefill and verify with the sigmoid-gated RMSNorm fused into the output epilogue ----
    ni = inputs.norm_inputs(T, H, seed=1100)
    pnorm = kda.OutputNorm(bf16_dev(ni.gate, device), f32_dev(ni.weight, device), ni.eps,
                           torch.empty((T, H), dtype=torch.float32, device=device))
    for _ in range(3):
        dev.run(out=out, final_state=final, workspace=ws, stream=stream, norm=pnorm)
    n_steps = max(3, min(args.steps, 200))
    n0 = torch.cuda.Event(enable_timing=True)
    n1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    n0.record(stream)
    for _ in range(n_steps):
        dev.run(out=out, final_state=final, workspace=ws, stream=stream, norm=pnorm)
    n1.record(stream)
    torch.cuda.synchronize(device)
    pn_us = n0.elapsed_time(n1) * 1e3 / n_steps
    pn_bytes = alg + T * H * NORM_BYTES_PER_ROW
    vni = inputs.norm_inputs(vin.B * vin.T, H, seed=1101)
    vnorm = kda.OutputNorm(bf16_dev(vni.gate, device), f32_dev(vni.weight, device), vni.eps,
                           torch.empty((vin.B * vin.T, H), dtype=torch.float32, device=device))
    vn_out = torch.empty((vin.B * vin.T, H, 128), dtype=torch.bfloat16, device=device)
    vn_inter = torch.empty((vin.B, vin.T, H, 128, 128), dtype=torch.float32, device=device)
    vn_us, vn_calls = graph_time_us(
        [lambda: vdev.run(out=vn_out, intermediate_states=vn_inter, workspace=ws, norm=vnorm)],
        max(3, min(args.steps, 200)))
    vn_bytes = verify_algorithmic_bytes(vin) + vin.B * vin.T * H * NORM_BYTES_PER_ROW
    assert kda.read_device_status(ws) == 0
    del vn_out, vn_inter, pnorm, vnorm
    gated = {
        "prefill": {"workload": inp.name, "us_per_layer": pn_us, "steps": n_steps,
                    "extra_us_vs_plain": pn_us - avg_launch_s * 1e6,
                    "roofline": {"bound": "hbm", "achieved": pn_bytes / (pn_us * 1e-6) / 1e9, "peak": peak,
                                 "unit": "GB/s", "frac": pn_bytes / (pn_us * 1e-6) / 1e9 / peak,
                                 "algorithmic_bytes": pn_bytes}},
        "verify": {"workload": vin.name, "us_per_layer": vn_us, "calls_timed": vn_calls,
                   "roofline": {"bound": "hbm", "achieved": vn_bytes / (vn_us * 1e-6) / 1e9, "peak": peak,
                                "unit": "GB/s", "frac": vn_bytes / (vn_us * 1e-6) / 1e9 / peak,
                                "algorithmic_bytes": vn_bytes}},
    }

    # ---- the same prefill and verify with the short causal convolutions of q, k, v fused into their prologues ----
    ci = inputs.conv_inputs(H, inp.pool.shape[0], seed=1200)
    pconv = kda.ShortConv(f32_dev(ci.weight, device), bf16_dev(ci.pool, device), ci.silu,
                          window_dense=torch.empty((inp.num_seqs, 3, 3, H, 128), dtype=torch.bfloat16, device=device))
    for _ in range(3):
        dev.run(out=out, final_state=final, workspace=ws, stream=stream, conv=pconv)
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    c0.record(stream)
    for _ in range(n_steps):
        dev.run(out=out, final_state=final, workspace=ws, stream=stream, conv=pconv)
    c1.record(stream)
    torch.cuda.synchronize(device)
    pc_us = c0.elapsed_time(c1) * 1e3 / n_steps
    pc_bytes = alg + 2 * inp.num_seqs * H * CONV_WINDOW_BYTES
    vci = inputs.conv_inputs(H, vin.pool.shape[0], seed=1201)
    vconv = kda.ShortConv(f32_dev(vci.weight, device), bf16_dev(vci.pool, device), vci.silu,
                          step_windows=torch.empty((vin.B, vin.T, 3, 3, H, 128), dtype=torch.bfloat16, device=device))
    vc_out = torch.empty((vin.B * vin.T, H, 128), dtype=torch.bfloat16, device=device)
    vc_inter = torch.empty((vin.B, vin.T, H, 128, 128), dtype=torch.float32, device=device)
    vc_us, vc_calls = graph_time_us(
        [lambda: vdev.run(out=vc_out, intermediate_states=vc_inter, workspace=ws, conv=vconv)],
        max(3, min(args.steps, 200)))
    vc_bytes = verify_algorithmic_bytes(vin) + vin.B * H * CONV_WINDOW_BYTES * (1 + vin.T)
    assert kda.read_device_status(ws) == 0
    del vc_out, vc_inter, pconv, vconv
    short_conv = {
        "prefill": {"workload": inp.name, "us_per_layer": pc_us, "steps": n_steps,
                    "extra_us_vs_plain": pc_us - avg_launch_s * 1e6,
                    "roofline": {"bound": "hbm", "achieved": pc_bytes / (pc_us * 1e-6) / 1e9, "peak": peak,
                                 "unit": "GB/s", "frac": pc_bytes / (pc_us * 1e-6) / 1e9 / peak,
                                 "algorithmic_bytes": pc_bytes}},
        "verify": {"workload": vin.name, "us_per_layer": vc_us, "calls_timed": vc_calls,
                   "roofline": {"bound": "hbm", "achieved": vc_bytes / (vc_us * 1e-6) / 1e9, "peak": peak,
                                "unit": "GB/s", "frac": vc_bytes / (vc_us * 1e-6) / 1e9 / peak,
                                "algorithmic_bytes": vc_bytes}},
    }

    # ---- one spec step: prefill segment + verify segment, outputs written by index into the layer output ----
    sdev = DeviceSpecStep(inputs.spec_step_2048x4_64x4(), device=device)
    sin = sdev.inp
    s_ws = sdev.workspace()
    s_out = sdev.new_out()
    s_inter = torch.empty((sin.verify.B, sin.verify.T, H, 128, 128), dtype=torch.float32, device=device)
    for _ in range(3):
        sdev.run(out=s_out, intermediate_states=s_inter, workspace=s_ws)
    s_steps = max(3, min(args.steps, 200))
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    s0.record(stream)
    for _ in range(s_steps):
        sdev.run(out=s_out, intermediate_states=s_inter, workspace=s_ws, stream=stream)
    s1.record(stream)
    torch.cuda.synchronize(device)
    assert kda.read_device_status(s_ws) == 0
    s_us = s0.elapsed_time(s1) * 1e3 / s_steps
    s_bytes = spec_step_algorithmic_bytes(sin)
    s_achieved = s_bytes / (s_us * 1e-6) / 1e9
    s_tokens = sin.prefill.total_tokens + sin.verify.B * sin.verify.T
    del sdev, s_ws, s_out, s_inter

    # ---- the other prefill workloads, each timed as its own call (median of per-call CUDA events) ----
    # (defined here; the main workload's fused-path record is taken after them)
    def time_prefill(pinp, steps, note=None, path=None):
        pdev = DevicePrefill(pinp, device=device)
        pws = pdev.workspace(device)
        pout = torch.empty((pinp.total_tokens, pinp.H, 128), dtype=torch.bfloat16, device=device)
        pfinal = None if pinp.final_to_pool else torch.empty((pinp.num_seqs, pinp.H, 128, 128), dtype=torch.float32,
                                                             device=device)

        def call():
            pdev.run(out=pout, final_state=pfinal, workspace=pws, stream=stream, path=path)

        for _ in range(3):
            call()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        torch.cuda.synchronize(device)
        for a, b in ev:
            a.record(stream)
            call()
            b.record(stream)
        torch.cuda.synchronize(device)
        assert kda.read_device_status(pws) == 0
        us = sorted(a.elapsed_time(b) * 1e3 for a, b in ev)
        med = statistics.median(us)
        # the same call captured in a CUDA graph and replayed: device time without the per-call host cost of the
        # binding and the launches (which dominates the eager figure of a tiny call)
        side = torch.cuda.Stream(device)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            call()
        stream.wait_stream(side)
        torch.cuda.synchronize(device)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            pdev.run(out=pout, final_state=pfinal, workspace=pws, path=path)
        graph.replay()
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(device)
        g0.record()
        for _ in range(steps):
            graph.replay()
        g1.record()
        torch.cuda.synchronize(device)
        graph_us = g0.elapsed_time(g1) * 1e3 / steps
        del graph
        nbytes = prefill_algorithmic_bytes(pinp)
        ach = nbytes / (med * 1e-6) / 1e9
        lens = pinp.cu_seqlens[1:] - pinp.cu_seqlens[:-1]
        rec = {"workload": pinp.name, "tokens": pinp.total_tokens, "sequences": pinp.num_seqs, "H": pinp.H,
               "longest_sequence": int(lens.max()), "chunks_of_longest": int((lens.max() + 63) // 64),
               "us_per_layer": med, "us_per_layer_min": us[0], "us_per_layer_max": us[-1], "calls_timed": steps,
               "us_per_layer_graph": graph_us,
               "tokens_per_s": pinp.total_tokens / (med * 1e-6),
               "roofline": {"bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
                            "algorithmic_bytes": nbytes},
               "l2": "inputs larger than L2" if nbytes > L2_BYTES else "fits in L2: launch-latency-bound"}
        if note:
            rec["note"] = note
        if path:
            rec["path"] = path
        return rec

    def fused_record(pinp, steps):
        """The same call on the fused one-kernel path (KDA_FUSED): every chunk's operands stay on chip."""
        r = time_prefill(pinp, steps, path="fused")
        rec = {k: r[k] for k in ("us_per_layer", "us_per_layer_graph", "tokens_per_s", "calls_timed")} | {
            "roofline_frac": r["roofline"]["frac"], "kernel": "prefill_fused_kernel (one launch)"}
        if pinp.name == WORKLOAD:   # DRAM bytes of one call from the committed ncu record (2048 x 8)
            rec["traffic"] = recorded_traffic("prefill_fused")
            rec["algorithmic_bytes"] = r["roofline"]["algorithmic_bytes"]
        return rec

    def two_pass_record(pinp, steps):
        """The same call with the two kernels on the plain schedule (KDA_TWO_PASS): the long workloads' default
        splits the longest sequences' state passes into segments that run beside later intra-chunk work."""
        r = time_prefill(pinp, steps, path="two_pass")
        return {k: r[k] for k in ("us_per_layer", "us_per_layer_graph", "tokens_per_s", "calls_timed")} | {
            "roofline_frac": r["roofline"]["frac"]}

    w_steps = max(20, min(args.steps, 200))
    workloads = {}
    for make in (inputs.tiny_prefill, inputs.prefill_8192x4, inputs.varlen_16384_plus_16):
        winp = make()
        workloads[winp.name] = time_prefill(winp, w_steps)
        workloads[winp.name]["fused_path"] = fused_record(winp, w_steps)
        if winp.total_tokens > 4096:
            workloads[winp.name]["two_pass_path"] = two_pass_record(winp, w_steps)
        if winp.name.startswith("prefill_16384"):
            # the long sequence of this workload alone: its state recurrence is one serial chain of 256 chunks per
            # head, the part of the workload that no number of SMs shortens (the pages quote 16384 x 1 as well)
            n0 = int(winp.cu_seqlens[1])
            long_inp = inputs.PrefillInputs(
                name="prefill_16384x1_h16 (the long sequence of prefill_16384+16varlen_h16 alone)",
                q=winp.q[:n0], k=winp.k[:n0], v=winp.v[:n0], g=winp.g[:n0], beta=winp.beta[:n0], A_log=winp.A_log,
                dt_bias=winp.dt_bias, lower_bound=winp.lower_bound, scale=winp.scale,
                cu_seqlens=winp.cu_seqlens[:2].copy())
            rec = time_prefill(long_inp, w_steps)
            rec["us_per_chunk"] = rec["us_per_layer"] / rec["chunks_of_longest"]
            rec["fused_path"] = fused_record(long_inp, w_steps)
            rec["two_pass_path"] = two_pass_record(long_inp, w_steps)
            workloads[winp.name]["long_sequence"] = rec
        if rank == 0 and not args.no_cpu_baseline and world == 1:
            workloads[winp.name]["cpu_baseline"] = cpu_baseline(winp, budget_s=5.0)
        del winp

    main_fused = fused_record(inp, w_steps)

    if rank != 0:
        return
    cpu = None if args.no_cpu_baseline or world > 1 else cpu_baseline(inp, budget_s=10.0)
    if cpu is not None:
        vrec["cpu_baseline"] = cpu_baseline_verify(vin)
    traffic = recorded_traffic("prefill")
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": value / (16384 / (PAGES_FLASHKDA_US * 1e-6)),
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "H": H, "d": 128, "tokens_per_step": T, "sequences": inp.num_seqs,
                   "initial_state": "64-slot pool by slot id", "final_state": "dense",
                   "l2": f"inputs larger than L2 ({alg / 1e6:.0f} MB algorithmic per step > 129 MB L2)",
                   "parallelism": f"replicas x{world}",
                   "vs_baseline_ref": "FlashKDA 49 us/layer at T=2048x8 on GB300 (vLLM PR #55737), context only"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "algorithmic_bytes": alg, "median_launch_us": med_launch_s * 1e6,
                     "avg_launch_us": avg_launch_s * 1e6,
                     "kernels": "chunk_intra_kernel + chunk_chain_kernel (one prefill call)",
                     "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else peak_kind},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps, "ms_per_step": e2e_ms / e2e_steps,
                "h2d_ms_per_step": h2d_ms, "d2h_ms_per_step": d2h_ms,
                "pipelining": "step i+1's host-to-device copies and step i-1's device-to-host copies on their own "
                              "streams overlap step i's call (double-buffered device buffers)"},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
        "fused_path": main_fused,
        "workloads": workloads,
        "verify": vrec,
        "verify_variants": vvariants,
        "spec_step": {"workload": sin.name, "us_per_layer": s_us, "steps": s_steps, "tokens": s_tokens,
                      "tokens_per_s": s_tokens / (s_us * 1e-6), "launches_per_call": 3,
                      "roofline": {"bound": "hbm", "achieved": s_achieved, "peak": peak, "unit": "GB/s",
                                   "frac": s_achieved / peak, "algorithmic_bytes": s_bytes}},
        "gated_norm": gated,
        "short_conv": short_conv,
        "commit": {"workload": vin.name + " (1..8 accepted per request)", "us_per_layer": c_us, "calls_timed": c_steps,
                   "roofline": {"bound": "hbm", "achieved": c_achieved, "peak": peak, "unit": "GB/s",
                                "frac": c_achieved / peak, "algorithmic_bytes": c_bytes}},
        "wall_s_timed_region": wall,
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
