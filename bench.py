#!/usr/bin/env python3
"""Benchmark of the verify-and-graft step on one GB300 (or N independent replicas).

One step = a1 prune + a2 graft + a3 mask + a4 tree attention + a5/a6 verify + a7 table
update for every request of the workload, issued through the C ABI on one stream with no
host synchronisation. The timed region replays a CUDA graph of K such steps; the inputs
rotate over several device copies whose total size is a multiple of the 129 MB L2, so
every step streams its K/V cache and logits from HBM.

Prints ONE JSON line. The GPU arm runs on exactly one GPU (it refuses WORLD_SIZE > 1
before touching CUDA); `--impl reference` times the CPU oracle instead (under torchrun,
rank 0 alone runs and prints it).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workload import CONFIGS, make_scenario  # noqa: E402

DEFAULT_CONFIG = 3   # the long-context workload (32K prefix) on which the HBM bar is stated
METRIC = "verify-and-graft steps/s on 1 GB300; tree-attn HBM GB/s as % of ~8 TB/s roofline"
# tree build, attention + combine, top-k (at T > 0 draws and top-k in one pass), walk + table
KERNELS_PER_STEP = 5
L2_BYTES = 129 * 2 ** 20
# Event record nodes end the programmatic overlap of the calls around them, so the timed
# graph brackets the attention call with events in one step out of ATTN_EVENT_EVERY only.
ATTN_EVENT_EVERY = 8  # one step in 8 has its attention call bracketed by events
ATTN_MIN_TIMED = 10   # bracketed attention calls per run, however few steps are timed


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), "measured"
    return 6800.0, "fallback"


def _tensor_peak():
    """Dense bf16 TFLOP/s: the measured burst figure (a kernel timed inside a short graph
    replay at full clock), else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if "bf16_tflops" in d:
            return d["bf16_tflops"], "measured (burst)"
    return 1900.0, "fallback (burst)"


def attn_flops(scn) -> int:
    """Algorithmic FLOPs of one gt_tree_attn call: Q K^T and P V for the g*N query rows of
    every (request, KV head) against every key the rows may see (prefix + tree),
    4 * rows * keys * d."""
    g = scn.Hq // scn.Hkv
    return sum(4 * g * scn.N * (int(P) + scn.N) * scn.d for P in scn.prefix_len) * scn.Hkv


def attn_bytes(scn) -> int:
    """Algorithmic bytes of one gt_tree_attn call: the K and V rows each request attends
    (prefix + tree), Q read once, O written once."""
    es = 2 if scn.dtype == "bf16" else 4
    kv = sum(int(P) + scn.N for P in scn.prefix_len) * scn.Hkv * scn.d * es * 2
    qo = 2 * scn.B * scn.N * scn.Hq * scn.d * es
    return kv + qo


def step_bytes(scn) -> int:
    """Algorithmic bytes of the whole step: attention bytes + logits + the tree arrays, the
    template, the table rows read by the graft and written by the update."""
    B, N = scn.B, scn.N
    logits = B * N * scn.V * 4
    tree = B * scn.Nin * 12 + B * N * (4 * 6 + 8)          # prune in, tree out, mask, pos, depth
    table = B * N * scn.k * 4 * 2 + len(scn.tpar) * 8       # graft reads + update writes
    verify = B * N * scn.k * 8 + B * N * 16
    return attn_bytes(scn) + logits + tree + table + verify


def rotation(scn):
    """(bytes of one input set, number of device copies the timed graph rotates over): the
    K/V cache, Q, the logits and the table of one set; enough sets that four L2 sizes pass
    between two uses of the same set."""
    es = 2 if scn.dtype == "bf16" else 4
    per_set = (2 * scn.K.size + scn.Q.size) * es + scn.B * scn.N * scn.V * 4 + \
        scn.table.size * 4
    return per_set, max(2, -(-4 * L2_BYTES // per_set))


def workload_config(scn, cid: int, temperature: float) -> dict:
    """The `config` object both arms print: what the workload is, nothing measured."""
    per_set, nsets = rotation(scn)
    return {"workload": scn.name, "config_id": cid, "B": scn.B, "temperature": temperature,
            "prefix_len": int(max(scn.prefix_len)), "slots": scn.N, "vocab": scn.V,
            "heads": f"{scn.Hq}/{scn.Hkv}x{scn.d}", "parallelism": "single GPU",
            "l2": f"inputs rotate over {nsets} device copies of {per_set / 1e6:.1f} MB "
                  f"(> L2 of {L2_BYTES / 2**20:.0f} MiB)",
            "step_bytes": step_bytes(scn)}


class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML (read-only queries) on a
    background thread while the timed region runs; falls back to nvidia-smi polling."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu_index: int, period_s: float = 0.002):
        import ctypes
        import threading
        self.samples, self.reasons, self.max_mhz = [], set(), None
        self._stop = threading.Event()
        self._thread = None
        self._nvml = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(gpu_index), ctypes.byref(h)) != 0:
                raise OSError("no NVML handle")
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            getr = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self._nvml = (nv, h, getr)
        except (OSError, AttributeError):
            self._nvml = None

        def run():
            nv, h, getr = self._nvml
            clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
            while not self._stop.is_set():
                if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                    self.samples.append(float(clk.value))
                if getr(h, ctypes.byref(rs)) == 0:
                    for bit, name in self.REASONS.items():
                        if rs.value & bit:
                            self.reasons.add(name)
                time.sleep(period_s)

        if self._nvml is not None:
            self._thread = threading.Thread(target=run, daemon=True)

    def start(self):
        if self._thread is not None:
            self._thread.start()
        return self

    def stop(self):
        if self._thread is None:
            return None
        self._stop.set()
        self._thread.join()
        if not self.samples:
            return None
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples),
                "source": "nvml"}


def _traffic_record(kernel_key: str, field: str = "bytes_per_launch"):
    """DRAM bytes per launch from a committed ncu summary, if the kernel's sources are
    unchanged since the capture (sha256 of ATTN_SOURCES), else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(kernel_key)
    if not rec:
        return None
    return rec.get(field) if rec.get("src_sha256") == _src_hash() else None


# the sources the attention kernels (tcgen05, SIMT, combine) are compiled from
ATTN_SOURCES = ("attn.cu", "attn_tc.cu", "attn_tc.cuh", "attn_common.cuh", "tc_ptx.cuh",
                "gt_internal.cuh", "launch.cuh")


def _src_hash(names=ATTN_SOURCES) -> str:
    """sha256 over the named CUDA sources (name and content, in the given order)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tree_speculative_decoding_parent_gb300", "csrc")
    for f in names:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()


# --------------------------------------------------------------------------------------
# CPU oracle timing (reference arm and cpu_baseline)
# --------------------------------------------------------------------------------------


def time_oracle(scn, steps: int, budget_s: float, temperature: float = 0.0, seed: int = 1):
    """Runs the oracle's whole step on the same workload; returns (steps/s, steps, seconds)."""
    import oracle
    tree = oracle.step_tree_phase(scn.parent_in, scn.tokens_in, scn.score_in,
                                  [scn.Nin] * scn.B, scn.keep, scn.thresh, scn.tpar, scn.trank,
                                  scn.R, scn.table, scn.prefix_len, scn.N, anchor=scn.anchor)
    logits = scn.logits(tree["parent"], tree["tokens"], tree["n_nodes"])
    dec = oracle.bf16_to_f64 if scn.dtype == "bf16" else (lambda a: np.asarray(a, np.float64))
    done, t0 = 0, time.perf_counter()
    table = scn.table
    while done < steps:
        tree = oracle.step_tree_phase(scn.parent_in, scn.tokens_in, scn.score_in,
                                      [scn.Nin] * scn.B, scn.keep, scn.thresh, scn.tpar,
                                      scn.trank, scn.R, table, scn.prefix_len, scn.N,
                                      anchor=scn.anchor)
        for b in range(scn.B):
            n, P = int(tree["n_nodes"][b]), int(scn.prefix_len[b])
            oracle.tree_attn(dec(scn.Q[b]), dec(scn.K[b][:, :P + n]), dec(scn.Vc[b][:, :P + n]),
                             tree["parent"][b], n, P, scn.scale)
        if temperature > 0:
            res = oracle.step_verify_sampled(tree, logits, table, scn.prefix_len, scn.k,
                                             temperature, seed, done)
        else:
            res = oracle.step_verify_phase(tree, logits, table, scn.prefix_len, scn.k)
        table = res["table"]
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return done / dt, done, dt


def run_reference(args, rank: int, world: int):
    if rank != 0:
        return None
    scn = make_scenario(args.config)
    # one untimed warm-up step (the oracle has no caches to fill)
    time_oracle(scn, 1, 0.0, args.temperature, args.seed)
    value, done, dt = time_oracle(scn, args.steps, args.ref_budget, args.temperature, args.seed)
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "steps/s",
        "n_gpus": world, "steps": done, "warmup": args.warmup, "ms_per_step": 1e3 * dt / done,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded generator of the five workload shapes)",
        "config": workload_config(scn, args.config, args.temperature),
        "cpu_baseline": {"value": value, "unit": "steps/s", "cores": cores, "kind": "oracle",
                         "sample": f"{done} whole steps of the same workload on the host CPU "
                                   f"(numpy float64; BLAS may use all {cores} cores)"},
        "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    return line


# --------------------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------------------


def run_gpu(args):
    import torch
    from tree_speculative_decoding_parent_gb300 import build, gt
    from tree_speculative_decoding_parent_gb300.step import (StepBuffers, StepShape, run_attn,
                                                             run_step, run_tree_build,
                                                             run_tree_phase, run_verify_commit,
                                                             run_verify_sample_commit)
    build.build()
    gt.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    scn = make_scenario(args.config)
    shape = StepShape(B=scn.B, Nin=scn.Nin, N=scn.N, V=scn.V, k=scn.k, Hq=scn.Hq, Hkv=scn.Hkv,
                      d=scn.d, Lcap=scn.Lcap, T=len(scn.tpar),
                      dtype=gt.GT_BF16 if scn.dtype == "bf16" else gt.GT_F32)
    bf16 = scn.dtype == "bf16"

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    def qkv(a):
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16) \
            if bf16 else torch.from_numpy(np.ascontiguousarray(a))
        return t.to(dev)

    base = dict(score_in=to_dev(scn.score_in), parent_in=to_dev(scn.parent_in),
                tokens_in=to_dev(scn.tokens_in), keep=to_dev(scn.keep), R=to_dev(scn.R),
                table=to_dev(scn.table), prefix_len=to_dev(scn.prefix_len),
                Q=qkv(scn.Q), K=qkv(scn.K), V=qkv(scn.Vc))
    if scn.thresh is not None:
        base["thresh"] = to_dev(scn.thresh)
    if scn.anchor is not None:
        base["anchor"] = to_dev(scn.anchor)
    if len(scn.tpar):
        base["tpar"], base["trank"] = to_dev(scn.tpar), to_dev(scn.trank)
    # plant the target logits on the tree this GPU path builds from the inputs
    buf = StepBuffers(shape, dev)
    run_tree_phase(buf, base)
    torch.cuda.synchronize()
    logits_np = scn.logits(buf.parent.cpu().numpy(), buf.tokens.cpu().numpy(),
                           buf.n_nodes.cpu().numpy())
    base["logits"] = to_dev(logits_np)
    per_set, nsets = rotation(scn)
    sets = [base] + [{k: v.clone() for k, v in base.items()} for _ in range(nsets - 1)]
    stream = torch.cuda.current_stream(dev)

    # eager warm-up (first calls set kernel attributes), then graphs
    run_step(buf, sets[0], scale=scn.scale, temperature=args.temperature, seed=args.seed)
    torch.cuda.synchronize()
    if int(buf.err.item()) != 0:
        raise RuntimeError(f"device error {gt.status_string(int(buf.err.item()))}")

    side = torch.cuda.Stream(dev)

    def event_pool(n: int):
        """n timing events, each recorded once (torch creates CUDA events lazily, and a graph
        can only record an event that exists)."""
        pool = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in pool:
            e.record(stream)
        torch.cuda.synchronize()
        return pool

    def capture(nsteps: int, event_every: int = 0, in_step: bool = False, ev_pool=()):
        """A graph of nsteps whole steps rotating over the input sets. event_every > 0: the
        attention call of every event_every-th step is bracketed by event records on the
        launch stream (which ends the programmatic overlap with the calls around it).
        in_step: every step's attention call is bracketed by event records on a side branch
        of the graph, forked after the tree build and joined after the attention's last
        kernel, so the launch stream's chain keeps its programmatic overlaps and the events
        mark the interval the call adds to the step."""
        g = torch.cuda.CUDAGraph()
        evs = []
        with torch.cuda.graph(g):
            s = torch.cuda.current_stream()
            for i in range(nsteps):
                inp = sets[i % nsets]
                run_tree_build(buf, inp, s)
                timed = event_every > 0 and i % event_every == 0
                if timed or in_step:
                    e0, e1 = ev_pool[2 * len(evs)], ev_pool[2 * len(evs) + 1]
                if timed:
                    gt.gt_event_record_external(e0, s)
                if in_step:
                    fork = torch.cuda.Event()
                    fork.record(s)
                    side.wait_event(fork)
                    gt.gt_event_record_external(e0, side)
                run_attn(buf, inp, s, scn.scale)
                if timed:
                    gt.gt_event_record_external(e1, s)
                if in_step:
                    join = torch.cuda.Event()
                    join.record(s)
                    side.wait_event(join)
                    gt.gt_event_record_external(e1, side)
                if timed or in_step:
                    evs.append((e0, e1))
                if args.temperature > 0:
                    run_verify_sample_commit(buf, inp, args.temperature, args.seed, i, s)
                else:
                    run_verify_commit(buf, inp, s)
            if in_step:
                s.wait_stream(side)  # every forked branch rejoins before the capture ends
        return g, evs

    # The timed graph times the attention call of every step on a side branch (no event node
    # sits on the launch stream's chain). A second graph of the same steps brackets one
    # attention call in ATTN_EVENT_EVERY on the launch stream itself (at least ATTN_MIN_TIMED
    # calls): those calls lose their overlap with the tree build, so they read slower.
    attn_steps = max(args.steps, ATTN_EVENT_EVERY * ATTN_MIN_TIMED)
    g_warm, _ = capture(max(args.warmup, 1))
    g_timed, step_evs = capture(args.steps, in_step=True, ev_pool=event_pool(2 * args.steps))
    g_attn, evs = capture(attn_steps, ATTN_EVENT_EVERY, ev_pool=event_pool(2 * attn_steps))
    g_warm.replay()
    torch.cuda.synchronize()
    clk = ClockSampler(torch.cuda.current_device())
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    replay_ms, in_step_by_replay = [], []
    clk.start()
    for _ in range(args.reps):
        torch.cuda.synchronize()
        t0.record(stream)
        g_timed.replay()
        t1.record(stream)
        torch.cuda.synchronize()
        replay_ms.append(t0.elapsed_time(t1))
        in_step_by_replay.append([a.elapsed_time(b) for a, b in step_evs])
    g_attn.replay()
    torch.cuda.synchronize()
    clocks = clk.stop()
    ms = statistics.median(replay_ms)
    errc = int(buf.err.item())
    if errc != 0:
        raise RuntimeError(f"device error {gt.status_string(errc)}")
    attn_ms = [a.elapsed_time(b) for a, b in evs]
    bracketed_avg_ms = sum(attn_ms) / len(attn_ms)
    # A graph's first launch records the first few side-branch events late (measured: the
    # first one to three steps of the first replay read about 2 us, every later replay none),
    # so the in-step samples come from the replays after the first when there are several.
    kept = in_step_by_replay[1:] if len(in_step_by_replay) > 1 else in_step_by_replay
    in_step_ms = [x for r in kept for x in r]
    attn_avg_ms = sum(in_step_ms) / len(in_step_ms)

    # ---- end to end through host buffers: H2D of the step's inputs, D2H of its result
    pin = lambda t: t.cpu().pin_memory()  # noqa: E731
    h_tree = {k: pin(base[k]) for k in ("score_in", "parent_in", "tokens_in", "keep", "R")}
    for key in ("thresh", "anchor"):
        if key in base:
            h_tree[key] = pin(base[key])
    h_q = pin(base["Q"])
    P = scn.prefix_len
    h_kv = [(pin(base["K"][b, :, P[b]:P[b] + scn.N]), pin(base["V"][b, :, P[b]:P[b] + scn.N]))
            for b in range(scn.B)]
    h_logits = pin(base["logits"])
    outs = ("acc_len", "out_tok", "path", "kv_src", "kv_dst")
    h_out = {k: torch.empty(getattr(buf, k).shape, dtype=torch.int32).pin_memory() for k in outs}
    h2d = sum(t.numel() * t.element_size() for t in list(h_tree.values()) + [h_q, h_logits]) + \
        sum(a.numel() * a.element_size() * 2 for a, _ in h_kv)
    d2h = sum(t.numel() * t.element_size() for t in h_out.values())
    inp = sets[0]

    copy_side = torch.cuda.Stream(dev)
    logits_in = torch.cuda.Event()

    def e2e_work():
        # the logits (most of the bytes) are needed only by the verify: they cross the host
        # link on a side stream while the small inputs arrive and the tree build and the
        # attention run; the verify waits for them
        # (the small inputs are queued first: copies on one engine run in order)
        main = torch.cuda.current_stream()
        for k, t in h_tree.items():
            inp[k].copy_(t, non_blocking=True)
        inp["Q"].copy_(h_q, non_blocking=True)
        for b in range(scn.B):
            inp["K"][b, :, P[b]:P[b] + scn.N].copy_(h_kv[b][0], non_blocking=True)
            inp["V"][b, :, P[b]:P[b] + scn.N].copy_(h_kv[b][1], non_blocking=True)
        copy_side.wait_stream(main)
        with torch.cuda.stream(copy_side):
            # in copies of at most 32 MB: one large copy replays slower from a graph
            dl, hl = inp["logits"].view(-1), h_logits.view(-1)
            step = 8 << 20  # floats
            for o in range(0, dl.numel(), step):
                dl[o:o + step].copy_(hl[o:o + step], non_blocking=True)
            logits_in.record(copy_side)
        run_tree_build(buf, inp, main)
        run_attn(buf, inp, main, scn.scale)
        main.wait_event(logits_in)
        if args.temperature > 0:
            run_verify_sample_commit(buf, inp, args.temperature, args.seed, 0, main)
        else:
            run_verify_commit(buf, inp, main)
        for k in outs:
            h_out[k].copy_(getattr(buf, k), non_blocking=True)

    def e2e_step():
        e2e_work()
        torch.cuda.synchronize()

    for _ in range(3):
        e2e_step()
    ne = max(5, min(args.steps, 50))

    def time_e2e(step_fn):
        torch.cuda.synchronize()
        te = time.perf_counter()
        for _ in range(ne):
            step_fn()
        return time.perf_counter() - te

    e2e_eager_s = time_e2e(e2e_step)
    # the same step (host-to-device copies, the calls, the read-back) captured once and
    # replayed per step with a host synchronisation, as a serving loop replays its decode
    # graph; steps stay strictly serial (a step's inputs never overlap the previous step)
    g_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_e2e):
        e2e_work()
    g_e2e.replay()
    torch.cuda.synchronize()

    def e2e_graph_step():
        g_e2e.replay()
        torch.cuda.synchronize()

    e2e_s = time_e2e(e2e_graph_step)

    breakdown = None
    if args.breakdown:
        breakdown = call_breakdown(torch, gt, buf, sets, scn, nsets, args.temperature, args.seed)

    peak, peak_kind = _peaks()
    ab = attn_bytes(scn)
    achieved = ab / (attn_avg_ms * 1e-3) / 1e9
    # the attention's bound: HBM below the measured ridge (flops per byte of the tensor peak
    # over the copy bandwidth), the tensor pipe above it
    tpeak, tpeak_kind = _tensor_peak()
    af = attn_flops(scn)
    tensor_bound = af / ab > tpeak * 1e12 / (peak * 1e9)
    if tensor_bound:
        t_achieved = af / (attn_avg_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": t_achieved, "peak": tpeak, "unit": "TFLOP/s",
                "frac": t_achieved / tpeak, "peak_kind": tpeak_kind,
                "algorithmic_flops_per_launch": af, "hbm_gbs_achieved": achieved}
    else:
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "peak_kind": peak_kind}
    value = args.steps / (ms * 1e-3)
    sb = step_bytes(scn)
    line = {
        "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": scn.dtype,
        "data": "synthetic (seeded generator of the five workload shapes)",
        "config": workload_config(scn, args.config, args.temperature),
        "value_spread": {"replays": len(replay_ms), "statistic": "median",
                         "steps_per_s": sorted(args.steps / (t * 1e-3) for t in replay_ms)},
        "step_byte_roofline_frac": sb / (ms / args.steps * 1e-3) / 1e9 / peak,
        "roofline": {**roof, "kernel": "gt_tree_attn (tcgen05/SIMT attention + combine)",
                     "flop_per_byte": af / ab,
                     "algorithmic_bytes_per_launch": ab,
                     "avg_launch_ms": attn_avg_ms,
                     "launch_ms_min_max": [min(in_step_ms), max(in_step_ms)],
                     "timed_launches": f"{len(in_step_ms)} calls: every step of "
                                       + ("every timed replay after the first (a graph's first "
                                          "launch records its first side-branch events late)"
                                          if len(in_step_by_replay) > 1 else "the timed replay")
                                       + ", from the end of the step's tree build to the end "
                                       "of the attention's last kernel (events on a side branch "
                                       "of the timed graph)",
                     "launch_stream_bracketed": {
                         "avg_ms": bracketed_avg_ms, "min_max_ms": [min(attn_ms), max(attn_ms)],
                         "frac": (af / (bracketed_avg_ms * 1e-3) / 1e12 / tpeak if tensor_bound
                                  else ab / (bracketed_avg_ms * 1e-3) / 1e9 / peak),
                         "calls": f"{len(attn_ms)} calls, one per {ATTN_EVENT_EVERY} steps of a "
                                  f"{attn_steps}-step graph, events on the launch stream (the "
                                  "call then loses its overlap with the tree build)"},
                     # DRAM bytes of one call (both kernels) recorded by ncu with the caches
                     # as the step leaves them; the flushed figure re-reads the partial rows
                     "traffic": _traffic_record(f"tree_attn/config{args.config}",
                                                "live_bytes_per_launch"),
                     "traffic_attn_kernel": _traffic_record(f"tree_attn/config{args.config}",
                                                            "live_attn_tc_kernel_bytes"),
                     "traffic_flushed": _traffic_record(f"tree_attn/config{args.config}")},
        "e2e": {"value": ne / e2e_s, "unit": "steps/s",
                "eager_value": ne / e2e_eager_s,
                "how": "pinned host inputs copied in (the logits on a side stream, overlapping "
                       "the tree build and the attention), the step's calls, results read back "
                       "and a host sync every step, replayed from one captured graph "
                       "(eager_value: the same calls issued one by one)",
                "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * KERNELS_PER_STEP,
        "clocks": clocks,
        "accepted_len_mean": float(buf.acc_len.float().mean().item()),
    }
    if breakdown is not None:
        line["breakdown_us"] = breakdown
        line["drafter_us"] = draft_timing(torch, gt)
    if not args.no_cpu_baseline:
        cv, cdone, cdt = time_oracle(scn, 1000, args.cpu_budget, args.temperature, args.seed)
        line["cpu_baseline"] = {
            "value": cv, "unit": "steps/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{cdone} whole steps of the same workload (~{cdt:.0f} s, numpy float64; "
                      "BLAS may use every core, the tree and top-k loops use one)",
            "single_thread": oracle_single_thread(args.config, args.cpu_budget,
                                                  args.temperature, args.seed)}
    return line


def _single_thread_child(cid, budget, temperature, seed, out):
    scn = make_scenario(cid)
    out.put(time_oracle(scn, 1000, budget, temperature, seed))


def oracle_single_thread(cid: int, budget: float, temperature: float, seed: int) -> dict:
    """The same oracle timing in a fresh process whose BLAS and OpenMP pools have one thread
    (the variables are read when numpy loads, so they are set for a spawned child)."""
    import multiprocessing as mp
    names = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {n: os.environ.get(n) for n in names}
    try:
        for n in names:
            os.environ[n] = "1"
        ctx = mp.get_context("spawn")
        q = ctx.Queue()
        p = ctx.Process(target=_single_thread_child, args=(cid, budget, temperature, seed, q))
        p.start()
        value, done, dt = q.get(timeout=budget + 600)
        p.join(timeout=60)
    finally:
        for n, v in saved.items():
            if v is None:
                os.environ.pop(n, None)
            else:
                os.environ[n] = v
    return {"value": value, "unit": "steps/s", "cores": 1,
            "sample": f"{done} whole steps (~{dt:.0f} s) with one BLAS/OpenMP thread"}


def draft_timing(torch, gt, reps: int = 20):
    """Device time of n-gram drafting steps (frontier select, n-gram draft, attach; three
    launches each), growing D = 5 steps from the root in a CUDA graph (schedule small,
    mid, small, mid, small; W = 10, m = 10, keys of up to 4 tokens) over 32,768-token
    histories. Returns microseconds per step for B = 1 and B = 16."""
    from workload import make_draft_scenario
    res = {}
    for B in (1, 16):
        ds = make_draft_scenario(B=B, L=32768, V=151936)
        N = ds.Nmax
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
        par0 = np.full((B, N), -1, np.int32)
        tok0 = np.full((B, N), -1, np.int32)
        tok0[:, 0] = ds.root
        sc0 = np.zeros((B, N), np.float32)
        sc0[:, 0] = 1.0
        init = dict(parent=t(par0), tokens=t(tok0), score=t(sc0), n=t(np.ones(B, np.int32)),
                    first_new=t(np.zeros(B, np.int32)),
                    visited=torch.zeros((B, N), dtype=torch.uint8, device="cuda"))
        cur = {k: v.clone() for k, v in init.items()}
        hist, hlen, cid, cp = t(ds.hist), t(ds.hist_len), t(ds.cache_id), t(ds.cache_p)
        fr = torch.empty((B, ds.W), dtype=torch.int32, device="cuda")
        nfr = torch.empty(B, dtype=torch.int32, device="cuda")
        kid = torch.empty((B, ds.W, ds.m), dtype=torch.int32, device="cuda")
        kp = torch.empty((B, ds.W, ds.m), dtype=torch.float32, device="cuda")
        match = torch.empty((B, ds.W, 2), dtype=torch.int32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")

        def grow(s):
            for mid in (0, 1, 0, 1, 0):
                gt.gt_frontier_select(cur["score"], cur["n"], B, N,
                                      None if mid else cur["first_new"],
                                      cur["visited"] if mid else None, ds.W, fr, nfr, err, s)
                gt.gt_ngram_draft(hist, hlen, B, hist.shape[1], cid, cp, ds.m, cur["parent"],
                                  cur["tokens"], cur["n"], N, fr, nfr, ds.W, ds.q_max, kid, kp,
                                  match, err, s)
                gt.gt_tree_attach(cur["parent"], cur["tokens"], cur["score"], cur["n"], B, N, fr,
                                  nfr, ds.W, kid, kp, ds.m, ds.V, cur["first_new"], err, s)

        grow(torch.cuda.current_stream())  # eager warm-up
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for e in (e0, e1):
            e.record()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            s = torch.cuda.current_stream()
            for k in cur:
                cur[k].copy_(init[k])
            gt.gt_event_record_external(e0, s)
            grow(s)
            gt.gt_event_record_external(e1, s)
        tot = 0.0
        for _ in range(reps):
            g.replay()
            torch.cuda.synchronize()
            tot += e0.elapsed_time(e1) * 1e3
        if int(err.item()) != 0:
            raise RuntimeError(f"drafting device error {gt.status_string(int(err.item()))}")
        res[f"B{B}"] = {"us_per_step": round(tot / reps / 5, 2),
                        "nodes_after_5_steps": int(cur["n"].float().mean().item())}
    return res


def call_breakdown(torch, gt, buf, sets, scn, nsets, temperature=0.0, seed=0, reps: int = 50):
    """Average device time of each C-ABI call of the step inside a CUDA graph: one graph
    per input set with an externally visible event between consecutive calls (the events
    also end the programmatic overlap between the calls, so the sum exceeds the step)."""
    from tree_speculative_decoding_parent_gb300.step import (run_attn, run_kv_commit,
                                                             run_tree_build, run_verify_commit,
                                                             run_verify_sample_commit)
    # the KV commit (compaction of the accepted rows) is timed too; it is not part of the step
    names = ["gt_tree_build", "gt_tree_attn",
             "gt_verify_sample_commit" if temperature > 0 else "gt_verify_commit",
             "gt_kv_commit (not in step)"]
    graphs = []
    for k in range(nsets):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
        for e in evs:
            e.record()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        inp = sets[k]
        with torch.cuda.graph(g):
            s = torch.cuda.current_stream()
            gt.gt_event_record_external(evs[0], s)
            run_tree_build(buf, inp, s)
            gt.gt_event_record_external(evs[1], s)
            run_attn(buf, inp, s, scn.scale)
            gt.gt_event_record_external(evs[2], s)
            if temperature > 0:
                run_verify_sample_commit(buf, inp, temperature, seed, k, s)
            else:
                run_verify_commit(buf, inp, s)
            gt.gt_event_record_external(evs[3], s)
            run_kv_commit(buf, inp, s)
            gt.gt_event_record_external(evs[4], s)
        graphs.append((g, evs))
    tot = [0.0] * len(names)
    for r in range(reps):
        g, evs = graphs[r % nsets]
        g.replay()
        torch.cuda.synchronize()
        for i in range(len(names)):
            tot[i] += evs[i].elapsed_time(evs[i + 1]) * 1e3
    return {n: round(t / reps, 2) for n, t in zip(names, tot)}


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1,
                    help="GPUs of the run; the GPU arm runs on exactly one")
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--reps", type=int, default=5,
                    help="replays of the timed graph; the line reports their median")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG, choices=sorted(CONFIGS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--breakdown", action="store_true",
                    help="also report the in-graph device time of each C-ABI call")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--temperature", type=float, default=0.0,
                    help="0: greedy verification; > 0: one target draw per node at this T")
    ap.add_argument("--seed", type=int, default=1, help="seed of the draws at T > 0")
    ap.add_argument("--ref-budget", type=float, default=60.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    args.reps = max(1, args.reps)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        # The attention kernel streams K/V through cluster-multicast TMA loads, which this
        # library runs only in single-GPU processes; the step is measured on one GPU.
        if world != 1 or args.gpus != 1:
            sys.stderr.write(f"bench.py: the GPU arm runs on exactly one GPU (got --gpus "
                             f"{args.gpus}, WORLD_SIZE {world}); nothing was run\n")
            sys.exit(2)
        line = run_gpu(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
