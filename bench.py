#!/usr/bin/env python
"""Decode-step benchmark: µs per layer at batch 1 and HBM GB/s over the
selected bytes, for the Deja Vu contextual-sparsity hot path on GB300.

One step = one decode token through all L stacked layers (predictor look-ahead
on a side stream, top-k, head-sparse attention with split-K, gather-fused
sparse MLP), captured once in a CUDA graph and replayed. Weights are seeded
random draws of the workload's shapes (no trained checkpoints); every step
reads far more than the 129 MB L2 (inputs larger than L2, no flush needed).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0). Multi-GPU: replicas only -- every rank decodes
its own copy of the workload on its own GPU; no data-path collective.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from contextual_sparsity_gb300 import build as dvbuild  # noqa: E402
from contextual_sparsity_gb300 import dv, synth, traffic  # noqa: E402

METRIC = "decode µs/layer at batch 1 and HBM GB/s over selected bytes vs 8 TB/s peak"
UNIT = "µs/layer"
NOMINAL_HBM = 8000.0
REPEATS = 5  # timed groups of steps; the headline is their median


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="opt-175b", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--keep-n", type=float, default=None)
    ap.add_argument("--keep-h", type=float, default=None)
    ap.add_argument("--layers", type=int, default=None)
    ap.add_argument("--n", type=int, default=None, help="cached tokens")
    ap.add_argument("--batch", type=int, default=None, help="sequences per step (1..4)")
    ap.add_argument("--sync", action="store_true", help="no look-ahead (predict each layer first)")
    ap.add_argument("--kv-dense", action="store_true",
                    help="composition workload: read the full cache (dense split-K baseline)")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--skip-inactive", action="store_true",
                    help="MLP streams fc2T rows only for neurons whose activation is above zero")
    ap.add_argument("--tuning", default=None,
                    help="main,side,main_ring_kb,side_ring_kb,attn,pdl,stage_kb (see dv_set_tuning)")
    ap.add_argument("--timeline", type=int, default=0,
                    help="print start/end of the first N launches of a profiled step to stderr")
    ap.add_argument("--decode-steps", type=int, default=0,
                    help="time T steps with a growing context, with and without the missing-KV "
                         "recompute")
    ap.add_argument("--input-corr", type=float, default=0.0,
                    help="--decode-steps: correlation of consecutive inputs (0 = independent)")
    ap.add_argument("--w4", action="store_true",
                    help="time the MLP block with fp16 and with 4-bit weight rows")
    ap.add_argument("--union-tc", action="store_true",
                    help="the MLP block over a batch's union at B = 4..64 (tensor cores from 8)")
    ap.add_argument("--step", action="store_true",
                    help="with --w4: whole decode steps with 4-bit weight rows vs fp16")
    ap.add_argument("--gate", action="store_true",
                    help="calibrate the latency gate on a context sweep and validate it")
    ap.add_argument("--gate-ctx", default="2048,8192,32768,131072",
                    help="sweep contexts the gate is calibrated on")
    ap.add_argument("--gate-val", default="4096,16384,65536",
                    help="held-out contexts the gate's predictions are checked on")
    return ap.parse_args()


def workload(a):
    over = {}
    if a.keep_n is not None:
        over["keep_N"] = a.keep_n
    if a.keep_h is not None:
        over["keep_H"] = a.keep_h
    if a.layers is not None:
        over["layers"] = a.layers
    if a.n is not None:
        over["n"] = a.n
    if a.batch is not None:
        over["B"] = a.batch
    return synth.workload(a.workload, **over)


def workload_name(w, lookahead=True):
    kv = f", KV keep {w.keep_KV:g}" if w.keep_KV < 1 else ""
    return (f"{w.name} (d {w.d}, {w.h}/{w.h_kv} heads x {w.dh}, FFN {w.F}, rank {w.r}, "
            f"{w.layers} layers, n {w.n}), neuron keep {w.keep_N:g}, head keep {w.keep_H:g}"
            f"{kv}, batch {w.B}, {'look-ahead' if lookahead else 'sync'} prediction")


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ---------------------------------------------------------------------------
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as tdist
        tdist.barrier()


def max_over_ranks(x, ws):
    if ws == 1:
        return x
    import torch.distributed as tdist
    dev = "cuda" if tdist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def job_figures(ms_total, steps, layers, ws, sel_bytes, pred_bytes):
    """Whole-job figures of N replicas that each ran `steps` steps of a
    `layers`-layer stack in ms_total (the slowest rank's time): µs per layer
    of the whole job (all ranks' layers in that time), per-replica µs per
    layer, and GB/s over selected and over all bytes summed over the ranks."""
    us_replica = ms_total * 1e3 / steps / layers
    us_job = us_replica / ws
    gbs_sel = ws * sel_bytes / (us_replica * 1e-6) / 1e9
    gbs_all = ws * (sel_bytes + pred_bytes) / (us_replica * 1e-6) / 1e9
    return {"us_layer_job": us_job, "us_layer_replica": us_replica, "gbs_selected": gbs_sel,
            "gbs_all": gbs_all, "layers_per_s": ws * layers * steps / (ms_total * 1e-3)}


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.lines = []
        self.proc = None

    def _gpu_id(self):
        try:
            u = str(torch.cuda.get_device_properties(self.dev).uuid)
            return u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES")
            return vis.split(",")[self.dev] if vis else str(self.dev)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms",
                 "100", "-i", self._gpu_id()], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for name, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# the workload on the GPU
# ---------------------------------------------------------------------------
class Model:
    def __init__(self, w, device, lookahead=True, seed=0, kv_dense=False, kept_inputs=False,
                 fill=False, extra_slots=0, w4=False, skip_inactive=False):
        self.w = w
        self.L = w.layers
        self.n = w.n
        self.n_max = w.n + 8 + extra_slots
        self.D = dv.dims(w.d, w.h, w.h_kv, w.dh, w.F, w.r, self.n_max)
        self.keep = dv.Keep(w.keep_N, w.keep_H, w.keep_KV)
        self.kN = traffic.k_of(w.keep_N, w.F)
        self.kH = traffic.k_of(w.keep_H, w.h_kv)
        self.W = [synth.layer_weights(w, l, seed=seed, device=device) for l in range(self.L)]
        if w4:
            # "Deja Vu" 5.2, Table 7 (W4A16): the projection and MLP rows as
            # packed 4-bit rows; the predictor stays fp16
            for W in self.W:
                for k in ("Wq", "Wk", "Wv", "WoT", "fc1", "fc2T"):
                    W[k] = dv.quantize_w4(W[k])
            torch.cuda.synchronize()
            torch.cuda.empty_cache()
        self.K, self.V = [], []
        for l in range(self.L):
            k, v = synth.kv_cache(w, l, self.n_max, seed=seed, device=device)
            self.K.append(k)
            self.V.append(v)
        # Composition with attention-scored KV selection: the scoring pass runs
        # once per layer (prefill time); every decode step then reads the
        # retained buffer through the same split-K kernel.
        self.retained = w.keep_KV < 1.0 and not kv_dense
        self.kv_flags = dv.DV_KV_RETAINED if self.retained else 0
        self.select_ms = None
        self.keys = w.n + 1
        flags_ws = dv.DV_KV_RESELECT if self.retained else 0
        self.ws = dv.workspace(self.D, w.B, flags_ws)
        if self.retained:
            self.b = int(w.n * w.keep_KV + 1e-9)
            self.b_max = self.b + 8
            self.keys = self.b + 1
            self.Kr, self.Vr, self.kp, self.kc, self.kvs = [], [], [], [], []
            qd = torch.zeros(w.h, w.dh, device=device)
            Hd = torch.zeros(w.h, w.dh, device=device)
            q_obs = []
            for l in range(self.L):
                Kr = torch.empty(w.h_kv, self.b_max, w.dh, dtype=torch.float16, device=device)
                Vr = torch.empty_like(Kr)
                kp = torch.zeros(w.h_kv, self.b_max, dtype=torch.int32, device=device)
                kc = torch.zeros(w.h_kv, dtype=torch.int32, device=device)
                kv = dv.kv_cache(self.K[l], self.V[l], Kr=Kr, Vr=Vr, kept_pos=kp, kept_count=kc,
                                 b_max=self.b_max)
                q_obs.append(synth.obs_queries(w, l, seed=seed, device=device))
                self.Kr.append(Kr); self.Vr.append(Vr); self.kp.append(kp); self.kc.append(kc)
                self.kvs.append(kv)

            def select(l):
                dv.kv_select_attn(qd, self.D, self.kvs[l], w.n, Hd, self.ws, q_obs=q_obs[l],
                                  obs_window=w.obs_window, n_sinks=w.n_sinks, smooth=w.smooth,
                                  kv_keep=w.keep_KV, flags=dv.DV_KV_RESELECT)
            select(0)  # warm (module load, tensor maps); it is repeated below
            torch.cuda.synchronize()
            e0, e1 = dv.event(True), dv.event(True)
            e0.record()
            for l in range(self.L):
                select(l)
            e1.record()
            torch.cuda.synchronize()
            self.select_ms = e0.elapsed_time(e1)
        elif kept_inputs or fill:
            # "Deja Vu" 4.2: a copy of each token's input and the missing-K/V
            # marks, so that later steps can recompute what this one skipped
            words = (w.h_kv + 31) // 32
            self.y_side = [torch.zeros(w.B, self.n_max, w.d, dtype=torch.float16, device=device)
                           for _ in range(self.L)]
            self.kv_miss = [torch.zeros(w.B, self.n_max, words, dtype=torch.int32, device=device)
                            for _ in range(self.L)]
            self.kvs = [dv.kv_cache(self.K[l], self.V[l], y_side=self.y_side[l],
                                    kv_missing=self.kv_miss[l]) for l in range(self.L)]
        else:
            self.kvs = [dv.kv_cache(self.K[l], self.V[l]) for l in range(self.L)]
        self.sets = [dv.sets(w.B, w.F, w.h_kv, self.kN, self.kH, device=device) for _ in range(2)]
        self.x = synth.hidden(w, seed=seed, device=device)
        self.y_tmp = torch.empty(2, w.B, w.d, dtype=torch.float16, device=device)
        self.y_out = torch.empty(w.B, w.d, dtype=torch.float16, device=device)
        self.side = torch.cuda.Stream(device=device)
        self.evf = dv.event()
        self.evj = dv.event()
        self.st = torch.zeros(1, dtype=torch.int32, device=device)
        flags = (dv.DV_LOOKAHEAD if lookahead else 0) | self.kv_flags
        if skip_inactive:
            flags |= dv.DV_SKIP_INACTIVE
        if w4:
            flags |= dv.DV_W4
        if fill:
            assert not self.retained, "the recompute reads the full cache"
            flags |= dv.DV_KV_FILL
        self.step = dv.Step(self.D, self.keep, self.W, self.kvs, [s for s, _ in self.sets],
                            self.ws, flags, self.side, self.evf, self.evj, dev_status=self.st)
        # the seeded draws above ran on the current stream; the step runs on others
        torch.cuda.synchronize()

    def capture(self, stream, profiler=None, x=None, n=None, warm=True):
        x = self.x if x is None else x
        n = self.n if n is None else n
        g = torch.cuda.CUDAGraph()
        stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            if warm:
                self.step(x, self.y_tmp, self.y_out, n, stream=stream)  # warm, outside capture
            torch.cuda.synchronize()
            n0 = dv.launch_count()
            if profiler:
                profiler.start()
            with torch.cuda.graph(g, stream=stream):
                self.step(x, self.y_tmp, self.y_out, n, stream=stream)
            if profiler:
                profiler.stop()
            per_step = dv.launch_count() - n0
        return g, per_step


# ---------------------------------------------------------------------------
# the oracle on the host (CPU baseline / reference arm)
# ---------------------------------------------------------------------------
def oracle_layer_seconds(w, budget_s, W=None, K=None, V=None, x=None, seed=0):
    """Time the fp64 oracle on one layer of the workload (predictor, top-k and
    the sparse layer in gather form), repeated until budget_s is spent."""
    import numpy as np

    import oracle

    oracle.build()
    if W is None:
        W = synth.layer_weights(w, 0, seed=seed)
        K, V = synth.kv_cache(w, 0, w.n + 1, seed=seed)
        x = synth.hidden(w, seed=seed)
    h = lambda t: t.detach().cpu().contiguous().numpy()
    Wh = {k: h(v) for k, v in W.items()}
    Kh, Vh, xh = h(K[0]), h(V[0]), h(x[0])
    kN, kH = traffic.k_of(w.keep_N, w.F), traffic.k_of(w.keep_H, w.h_kv)
    reps, t0 = 0, time.perf_counter()
    while True:
        s = oracle.predict(xh, Wh["P1"], Wh["P2"])
        selN = oracle.topk(s[: w.F], kN) if kN < w.F else np.arange(w.F)
        selH = oracle.topk(s[w.F:], kH) if kH < w.h_kv else np.arange(w.h_kv)
        oracle.layer(xh, Wh, Kh, Vh, w.n, selH, selN)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            return el / reps, reps


def run_reference(a):
    """The reference arm of this workload: the fp64 C oracle on the host, one
    layer of the stack per step (the metric is per layer). It runs exactly
    --warmup untimed and --steps timed single-layer steps, and reports the
    same config dict as the GPU arm."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np

    import oracle

    oracle.build()
    w = workload(a)
    W = synth.layer_weights(w, 0)
    K, V = synth.kv_cache(w, 0, w.n + 1)
    x = synth.hidden(w)
    h = lambda t: t.detach().cpu().contiguous().numpy()
    Wh = {k: h(v) for k, v in W.items()}
    Kh, Vh, xh = h(K[0]), h(V[0]), h(x[0])
    kN, kH = traffic.k_of(w.keep_N, w.F), traffic.k_of(w.keep_H, w.h_kv)

    def one_layer():
        s = oracle.predict(xh, Wh["P1"], Wh["P2"])
        selN = oracle.topk(s[: w.F], kN) if kN < w.F else np.arange(w.F)
        selH = oracle.topk(s[w.F:], kH) if kH < w.h_kv else np.arange(w.h_kv)
        oracle.layer(xh, Wh, Kh, Vh, w.n, selH, selN)

    for _ in range(a.warmup):
        one_layer()
    t0 = time.perf_counter()
    for _ in range(a.steps):
        one_layer()
    el = time.perf_counter() - t0
    val = el / a.steps * 1e6
    sample = (f"{a.steps} timed single-layer steps of {w.name} (predictor, top-k, sparse "
              f"attention and MLP in gather form), fp64 C oracle, one thread")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(val, 2), "unit": UNIT,
        "n_gpus": a.gpus, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": round(val / 1e3, 3), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "step": "one layer of the stack on the host (the metric is per layer)",
        "timed_region_s": round(el, 3),
        "config": config_dict(w, not a.sync, a.gpus),
        "cpu_baseline": {"value": round(val, 2), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample, "host_cpus": os.cpu_count()},
        "e2e": {"value": round(val, 2), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }))


def config_dict(w, lookahead, wsz):
    """The workload as both arms report it."""
    step_gb = sum(traffic.layer_bytes(w)) * w.layers / 1e9
    return {"workload": workload_name(w, lookahead), "layers": w.layers, "batch": w.B,
            "n_cached": w.n, "keep_neuron": w.keep_N, "keep_head": w.keep_H,
            "parallelism": "replicas" if wsz > 1 else "single GPU",
            "l2": (f"inputs larger than L2 (every step streams "
                   f"~{step_gb:.1f} GB)" if step_gb > 0.129 else
                   f"inputs fit in L2 (every step streams ~{step_gb * 1e3:.1f} MB)")}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# Source files each timed kernel is built from: a traffic record taken by ncu
# stays valid while these are unchanged.
KERNEL_SOURCES = {
    "k_stream<KIND_QKV>": ["k_stream.cu", "dv_common.cuh", "dv_internal.h"],
    "k_stream<KIND_WO>": ["k_stream.cu", "dv_common.cuh", "dv_internal.h"],
    "k_stream<KIND_MLP>": ["k_stream.cu", "dv_common.cuh", "dv_internal.h"],
    "k_splitk": ["k_attn.cu", "dv_common.cuh", "dv_internal.h"],
}


def traffic_record(kernel):
    """ncu DRAM bytes per launch of `kernel`, if the capture in profiles/ was
    taken on the kernel's current source (else None)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as f:
            j = json.load(f)
    except Exception:
        return None
    rec = j.get(kernel)
    if not rec:
        return None
    return rec["bytes_per_launch"] if rec.get("source_sha") == source_sha(kernel) else None


def source_sha(kernel):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "contextual_sparsity_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def run_ours(a):
    wsz, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dvbuild.build()
    dv.lib()
    if a.tuning:
        dv.set_tuning(*[int(x) for x in a.tuning.split(",")])
    w = workload(a)
    lookahead = not a.sync
    m = Model(w, dev, lookahead=lookahead, kv_dense=a.kv_dense, skip_inactive=a.skip_inactive)
    stream = torch.cuda.Stream(device=dev)
    g, per_step = m.capture(stream)
    torch.cuda.synchronize()

    for _ in range(max(3, a.warmup)):
        g.replay()
    torch.cuda.synchronize()
    # Exactly a.steps replays in one timed region; events at the boundaries of
    # REPEATS equal groups of steps inside it give the median over repeats.
    n_rep = max(1, min(REPEATS, a.steps))
    bounds = [a.steps * i // n_rep for i in range(n_rep + 1)]
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_rep + 1)]
    with ClockSampler(local) as clk:
        barrier(wsz)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            ev[0].record(stream)
            for i in range(n_rep):
                for _ in range(bounds[i + 1] - bounds[i]):
                    g.replay()
                ev[i + 1].record(stream)
        torch.cuda.synchronize()
        barrier(wsz)
    ms_total = max_over_ranks(ev[0].elapsed_time(ev[-1]), wsz)
    ms_step = ms_total / a.steps
    group_ms_step = [max_over_ranks(ev[i].elapsed_time(ev[i + 1]), wsz) / (bounds[i + 1] - bounds[i])
                     for i in range(n_rep)]
    median_ms_step = statistics.median(group_ms_step)
    assert m.st.item() == 0, f"device status {m.st.item()}"

    union = None
    if w.B > 1:
        # the union sizes the step produced (the two set buffers hold the
        # last two layers' sets)
        c = [t["ucnt"].cpu().tolist() for _, t in m.sets]
        uN = sum(x[0] for x in c) / 2 if w.keep_N < 1 else w.F
        uH = sum(x[1] for x in c) / 2 if w.keep_H < 1 else w.h_kv
        union = (uN, uH)
    sel, pred = traffic.layer_bytes(w, keys=m.keys, union=union)
    skip = None
    if a.skip_inactive:
        # the fc2T rows the MLP streamed (selected neurons with a positive
        # activation), counted on the device over one replay of the step
        cnt = torch.zeros(1, dtype=torch.int32, device=dev)
        dv.count_active(cnt)
        gc, _ = m.capture(stream, warm=False)
        dv.count_active(None)
        gc.replay()
        torch.cuda.synchronize()
        active = cnt.item() / w.layers / w.B
        kN_rows = union[0] if union else m.kN
        read = sel - (kN_rows - active) * w.d * 2
        skip = {"active_rows_per_layer": round(active, 1), "selected_rows_per_layer": kN_rows,
                "read_bytes_per_layer": round(read),
                "gbs_read": round(read / (median_ms_step * 1e3 / w.layers / wsz * 1e-6) / 1e9, 1)}
    # the headline: the median over the repeats (each of steps/REPEATS steps)
    job = job_figures(median_ms_step * a.steps, a.steps, w.layers, wsz, sel, pred)
    mean_us_layer = ms_total * 1e3 / a.steps / w.layers / wsz
    us_layer = job["us_layer_replica"]
    gbs_sel, gbs_all = job["gbs_selected"], job["gbs_all"]
    print(f"[bench] {us_layer:.2f} us/layer, {gbs_sel:.0f} GB/s selected, {gbs_all:.0f} GB/s all, "
          f"{per_step} launches/step", file=sys.stderr, flush=True)

    # Per-kernel durations: a second graph of the same step with every launch
    # bracketed by CUDA events on its own stream, replayed after warm-up.
    prof = dv.Profiler(cap=8 * per_step + 64)
    gp, _ = m.capture(stream, profiler=prof)
    for _ in range(max(3, a.warmup)):
        gp.replay()
    with torch.cuda.stream(stream):
        for _ in range(20):
            gp.replay()
    torch.cuda.synchronize()
    if a.timeline:
        t0 = prof.events[0]
        for i in range(min(a.timeline, prof.n)):
            tag = dv.TAGS.get(prof._tags[i], "?")
            b, e = t0.elapsed_time(prof.events[2 * i]), t0.elapsed_time(prof.events[2 * i + 1])
            print(f"[timeline] {i:4d} {tag:9s} {b * 1e3:9.2f} {e * 1e3:9.2f} {(e - b) * 1e3:8.2f}",
                  file=sys.stderr)
    per_kind = {}
    for tag, ms in prof.durations_ms():
        per_kind.setdefault(tag, []).append(ms * 1e3)
    kernel_us = {k: round(sum(v) / len(v), 2) for k, v in per_kind.items()}
    kernel_launches = {k: len(v) for k, v in per_kind.items()}
    G = w.h // w.h_kv
    # the QKV launch also streams the next layer's first predictor layer
    # (r rows of d) when predicting ahead
    p1_rows = (w.r if (lookahead and (w.keep_N < 1 or w.keep_H < 1) and w.layers > 1 and w.B == 1)
               else 0)
    kH_e, kN_e = (union[1], union[0]) if union else (m.kH, m.kN)
    algo = {
        "qkv": traffic.qkv_bytes(w.d, G, w.dh, kH_e) + traffic.p1_bytes(w.d, p1_rows),
        "wo": traffic.wo_bytes(w.d, G, w.dh, kH_e),
        "mlp": traffic.mlp_bytes(w.d, kN_e),
        "splitk": w.B * traffic.kv_bytes(w.dh, kH_e, m.keys),
    }
    totals = {k: sum(v) for k, v in per_kind.items()}
    dom = max(algo, key=lambda k: totals.get(k, 0.0))
    peak, peak_src = peaks()
    ach = algo[dom] / (kernel_us[dom] * 1e-6) / 1e9
    names = {"qkv": "k_stream<KIND_QKV>", "wo": "k_stream<KIND_WO>", "mlp": "k_stream<KIND_MLP>",
             "splitk": "k_splitk"}
    roof = {"bound": "hbm", "kernel": names[dom], "achieved": round(ach, 1), "peak": peak,
            "unit": "GB/s", "frac": round(ach / peak, 4), "peak_source": peak_src,
            "algorithmic_bytes_per_launch": algo[dom], "avg_launch_us": kernel_us[dom],
            "traffic": traffic_record(names[dom])}

    # End to end through the public API: every step copies its input from
    # pinned host memory, runs dv_decode_step (all layers) and copies the
    # result back, and the host waits for that result. Reported as a serving
    # caller would run it (the three calls captured once in a CUDA graph,
    # replayed per step) and, beside it, with dv_decode_step called eagerly.
    e2e = None
    if not a.no_e2e:
        hin = torch.empty(w.B, w.d, dtype=torch.float16).pin_memory()
        hin.copy_(m.x.cpu())
        hout = torch.empty(w.B, w.d, dtype=torch.float16).pin_memory()
        xin = torch.empty_like(m.x)

        def one_step():
            xin.copy_(hin, non_blocking=True)
            m.step(xin, m.y_tmp, m.y_out, m.n, stream=stream)
            hout.copy_(m.y_out, non_blocking=True)

        def timed(run):
            with torch.cuda.stream(stream):
                for _ in range(3):
                    run()
                stream.synchronize()
                barrier(wsz)
                t0 = time.perf_counter()
                for _ in range(a.e2e_steps):
                    run()
                    stream.synchronize()
                el = time.perf_counter() - t0
            return max_over_ranks(el, wsz) / a.e2e_steps * 1e6 / w.layers / wsz

        ge = torch.cuda.CUDAGraph()
        stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            one_step()
            stream.synchronize()
            with torch.cuda.graph(ge, stream=stream):
                one_step()
        us_graph = timed(ge.replay)
        us_eager = timed(one_step)
        assert m.st.item() == 0, f"device status {m.st.item()}"
        e2e = {"value": round(us_graph, 2), "unit": UNIT,
               "h2d_bytes_per_step": hin.numel() * 2, "d2h_bytes_per_step": hout.numel() * 2,
               "steps": a.e2e_steps,
               "api": "dv_decode_step with the pinned H2D input copy and the D2H result copy, "
                      "captured once in a CUDA graph, replayed per step, host waits per step",
               "eager_value": round(us_eager, 2),
               "eager_api": "dv_decode_step called per step (one C-ABI call, all layers)"}

    cpu = None
    if rank == 0 and wsz == 1 and not a.no_cpu_baseline:
        W0 = {k: v for k, v in m.W[0].items()}
        sec, reps = oracle_layer_seconds(w, a.cpu_seconds, W0, m.K[0], m.V[0], m.x)
        cpu = {"value": round(sec * 1e6, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{reps} repeats of one {w.name} layer (predictor, top-k, sparse "
                         f"attention and MLP in gather form), fp64 C oracle, one thread",
               "host_cpus": os.cpu_count()}

    if rank != 0:
        return
    out = {
        "metric": METRIC, "value": round(job["us_layer_job"], 2), "unit": UNIT, "n_gpus": wsz,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(ms_step, 4),
        "timing": {"repeats": n_rep, "steps_per_repeat": [bounds[i + 1] - bounds[i]
                                                          for i in range(n_rep)],
                   "value_is": "median over the repeats of their mean step time, per layer",
                   "us_layer_per_repeat": [round(t * 1e3 / w.layers / wsz, 2)
                                           for t in group_ms_step],
                   "us_layer_mean_all_steps": round(mean_us_layer, 2),
                   "timed_region_ms": round(ms_total, 3)},
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "accumulate": "f32", "data": "synthetic (seeded random weights of the workload's shapes)",
        "config": config_dict(w, lookahead, wsz),
        "selected_bytes_per_layer": round(sel), "predictor_bytes_per_layer": pred,
        "union_sizes": ({"neurons": union[0], "units": union[1]} if union else None),
        "kv": ({"mode": "retained", "keep": w.keep_KV, "budget": m.b, "keys_read": m.keys,
                "selection_ms_all_layers": round(m.select_ms, 3)} if m.retained else
               {"mode": "full cache", "keys_read": m.keys}),
        "gbs_selected": round(gbs_sel, 1),
        "frac_of_8tbs_selected": round(gbs_sel / (wsz * NOMINAL_HBM), 4),
        "gbs_all_traffic": round(gbs_all, 1),
        "frac_of_measured_hbm_selected": round(gbs_sel / (wsz * peak), 4),
        "us_layer_per_replica": round(us_layer, 2),
        "layers_per_s_total": round(job["layers_per_s"], 1),
        "skip_inactive": skip,
        "roofline": roof, "kernel_us": kernel_us, "kernel_launches_per_step": kernel_launches,
        "gpu_launches": per_step * a.steps, "launches_per_step": per_step,
        "clocks": clk.summary(), "e2e": e2e, "cpu_baseline": cpu,
    }
    print(json.dumps(out))


# ---------------------------------------------------------------------------
# latency gate: calibrate on a context sweep, validate, dispatch a request mix
# ---------------------------------------------------------------------------
GATE_KEEP = {  # (keep_N, keep_H, keep_KV) of each mode over the workload's own keeps
    dv.MODE_DENSE: lambda w: (1.0, 1.0, 1.0),
    dv.MODE_ACT: lambda w: (w.keep_N, w.keep_H, 1.0),
    dv.MODE_KV: lambda w: (1.0, 1.0, w.keep_KV),
    dv.MODE_COMPOSED: lambda w: (w.keep_N, w.keep_H, w.keep_KV),
}

# Requests of a mixed workload ("Where Activation Sparsity and KV-Cache
# Sparsity Cross in LLM Decoding" §5.4, App. I: chat turns, questions over long
# documents, agent loops): (context, decode steps, count).
GATE_MIX = [(2048, 256, 6), (4096, 128, 6), (8192, 64, 4), (16384, 64, 4), (32768, 256, 3),
            (65536, 128, 2), (131072, 256, 2)]


def _time_mode(w, dev, steps, warmup):
    """Per-layer µs of one graph-replayed decode step, and the scoring pass per
    layer (modes that select KV)."""
    m = Model(w, dev, lookahead=True, kv_dense=w.keep_KV >= 1.0)
    stream = torch.cuda.Stream(device=dev)
    g, _ = m.capture(stream)
    for _ in range(max(3, warmup)):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    assert m.st.item() == 0, f"device status {m.st.item()}"
    us = e0.elapsed_time(e1) * 1e3 / (steps * w.layers)
    sel = (m.select_ms * 1e3 / w.layers) if m.select_ms is not None else 0.0
    del m, g
    torch.cuda.empty_cache()
    return us, sel


def _measured_crossing(ctx, ta, tb):
    """Between the last context where a leads and the first where b leads,
    the linear zero of t_a - t_b (None if neither overtakes the other)."""
    for i in range(len(ctx) - 1):
        d0, d1 = ta[i] - tb[i], ta[i + 1] - tb[i + 1]
        if (d0 < 0 <= d1) or (d0 > 0 >= d1):
            return ctx[i] + d0 / (d0 - d1) * (ctx[i + 1] - ctx[i])
    return None


def run_multistep(a):
    """T decode steps with a growing context (n, n + 1, ..., n + T - 1), a new
    input per step, the look-ahead predictor choosing every step's sets: with
    and without the recompute of the missing K/V ("Deja Vu" 4.2)."""
    import numpy as np
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    dvbuild.build()
    dv.lib()
    w = workload(a)
    T = a.decode_steps
    # inputs x_t = rho x_{t-1} + sqrt(1 - rho^2) e_t: rho 0 gives independent
    # tokens (the predictor's sets nearly independent from step to step), rho
    # near 1 gives neighbouring tokens alike (overlapping sets, fewer holes)
    rho = a.input_corr
    xs = [synth.hidden(w, seed=1000, device=dev)]
    for t in range(1, T):
        e = synth.hidden(w, seed=1000 + t, device=dev).float()
        xs.append((rho * xs[-1].float() + (1.0 - rho * rho) ** 0.5 * e).half())
    passes = max(1, a.steps // T)
    res = {}
    for fill in (False, True):
        m = Model(w, dev, lookahead=not a.sync, kept_inputs=True, fill=fill, extra_slots=T)
        stream = torch.cuda.Stream(device=dev)
        graphs = [m.capture(stream, x=xs[t], n=w.n + t, warm=(t == 0))[0] for t in range(T)]
        for _ in range(max(1, a.warmup // T + 1)):
            for g in graphs:
                g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(passes):
                for g in graphs:
                    g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        assert m.st.item() == 0, f"device status {m.st.item()}"
        res["fill" if fill else "no_fill"] = e0.elapsed_time(e1) * 1e3 / (passes * T * w.layers)
        if not fill:
            # share of the units a step selects that the step before skipped
            # (each has at least one row to recompute); without the recompute
            # the marks keep every step's skips
            marks = torch.stack([k[:, w.n:w.n + T] for k in m.kv_miss]).cpu().numpy()
            bits = np.unpackbits(marks.view(np.uint8), axis=-1, bitorder="little")[..., :w.h_kv]
            sel_now, skip_prev = bits[:, :, 1:] == 0, bits[:, :, :-1] == 1
            res["hole_rate"] = round(float((sel_now & skip_prev).sum()) / float(sel_now.sum()), 3)
        # per-kernel times of the last step, replayed after the T - 1 before it
        prof = dv.Profiler(cap=64 * w.layers + 64)
        gp, _ = m.capture(stream, profiler=prof, x=xs[T - 1], n=w.n + T - 1, warm=False)
        for _ in range(3):
            for g in graphs[:-1]:
                g.replay()
            gp.replay()
        torch.cuda.synchronize()
        per_kind = {}
        for tag, ms in prof.durations_ms():
            per_kind.setdefault(tag, []).append(ms * 1e3)
        res["kernel_us_" + ("fill" if fill else "no_fill")] = {
            k: round(sum(v) / len(v), 2) for k, v in per_kind.items()}
        del m, graphs, gp
        torch.cuda.empty_cache()
        print(f"[multistep] {'fill' if fill else 'no fill'}: "
              f"{res['fill' if fill else 'no_fill']:.2f} us/layer", file=sys.stderr, flush=True)
    out = {"metric": "decode_steps_missing_kv", "workload": workload_name(w, not a.sync),
           "data": "synthetic", "decode_steps": T, "passes": passes, "input_corr": rho,
           "hole_rate": res.get("hole_rate"),
           "us_per_layer": {"no_fill": round(res["no_fill"], 2), "fill": round(res["fill"], 2)},
           "fill_cost_us_per_layer": round(res["fill"] - res["no_fill"], 2),
           "kernel_us": {"no_fill": res["kernel_us_no_fill"], "fill": res["kernel_us_fill"]}}
    print(json.dumps(out))


def run_union_tc(a):
    """The MLP block of a batch over the union of its sequences' neuron sets:
    B = 4 on the CUDA-core streaming kernel, B = 8..64 on the tensor cores
    ("Deja Vu" 5.2, App. C.1); sets drawn independently at the workload's keep."""
    import numpy as np
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    dvbuild.build()
    dv.lib()
    w = workload(a)
    kN = traffic.k_of(w.keep_N, w.F)
    W = synth.layer_weights(w, 0, device=dev)
    W = {k: W[k] for k in ("fc1", "fc2T", "b1", "ln2_g", "ln2_b") if k in W}
    torch.cuda.empty_cache()
    D = dv.dims(w.d, w.h, w.h_kv, w.dh, w.F, w.r, 8)
    stream = torch.cuda.Stream(device=dev)
    pk, pk_src = peaks()
    rows = []
    for B in (4, 8, 16, 32, 64):
        rng = np.random.default_rng(B)
        U = np.unique(np.concatenate([rng.choice(w.F, kN, replace=False) for _ in range(B)]))
        Ud = torch.from_numpy(U.astype(np.int32)).to(dev)
        x = synth.hidden(w, B=B, seed=7, device=dev)
        out = torch.empty(B, w.d, dtype=torch.float16, device=dev)
        if B == 4:
            ws = dv.workspace(D, B)
            run = lambda: dv.sparse_mlp(x, D, W, Ud, len(U), out, ws, stream=stream)
        else:
            ws = dv.union_mlp(x, D, W, Ud, len(U), out, stream=stream)
            run = lambda: dv.union_mlp(x, D, W, Ud, len(U), out, ws=ws, stream=stream)
        with torch.cuda.stream(stream):
            for _ in range(max(3, a.warmup)):
                run()
        torch.cuda.synchronize()
        reps = max(5, a.steps)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                run()
            e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / reps
        # per-launch durations of one more call, each launch between events
        prof = dv.Profiler(cap=16)
        prof.start()
        with torch.cuda.stream(stream):
            run()
        prof.stop()
        torch.cuda.synchronize()
        launch_us = [round(ms * 1e3, 2) for _, ms in prof.durations_ms()]
        by = traffic.mlp_bytes(w.d, len(U))
        rows.append({"B": B, "union": int(len(U)), "union_frac": round(len(U) / w.F, 3),
                     "us_per_block": round(us, 2), "us_per_sequence": round(us / B, 2),
                     "weight_bytes": by, "gbs": round(by / us / 1e3, 1),
                     "frac": round(by / us / 1e3 / pk, 3), "launch_us": launch_us,
                     "kernel": "k_stream<KIND_MLP> (CUDA cores)" if B == 4 else
                     "tcgen05 (TMEM accumulators, rows gathered by TMA gather4)"})
        print(f"[union] B {B}: |U| {len(U)} ({len(U) / w.F:.2f} F), {us:.1f} us", file=sys.stderr,
              flush=True)
    print(json.dumps({"metric": "union_mlp_block", "workload": workload_name(w), "data": "synthetic",
                      "neuron_keep": w.keep_N, "peak_gbs": pk, "peak_source": pk_src,
                      "rows": rows}))


def run_w4_step(a):
    """Whole decode steps of the workload with fp16 weights and with 4-bit
    projection and MLP rows (W4A16), same sets of rows, same graph replay."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    dvbuild.build()
    dv.lib()
    w = workload(a)
    res = {}
    for name in ("fp16", "w4"):
        m = Model(w, dev, lookahead=not a.sync, w4=(name == "w4"))
        stream = torch.cuda.Stream(device=dev)
        g, per_step = m.capture(stream)
        for _ in range(max(3, a.warmup)):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(a.steps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        assert m.st.item() == 0, f"device status {m.st.item()}"
        res[name] = e0.elapsed_time(e1) * 1e3 / (a.steps * w.layers)
        print(f"[w4-step] {name}: {res[name]:.2f} us/layer, {per_step} launches/step",
              file=sys.stderr, flush=True)
        del m, g
        torch.cuda.empty_cache()
    sel, _ = traffic.layer_bytes(w)
    sel4 = traffic.layer_bytes_w4(w)
    print(json.dumps({"metric": "decode_step_w4a16", "workload": workload_name(w, not a.sync),
                      "data": "synthetic", "steps": a.steps,
                      "us_per_layer": {k: round(v, 2) for k, v in res.items()},
                      "selected_bytes": {"fp16": sel, "w4": sel4},
                      "gbs_selected": {"fp16": round(sel / res["fp16"] / 1e3, 1),
                                       "w4": round(sel4 / res["w4"] / 1e3, 1)},
                      "speedup": round(res["fp16"] / res["w4"], 3)}))


def run_w4(a):
    """The MLP block with fp16 rows and with 4-bit rows (W4A16, "Deja Vu"
    5.2, Table 7) at the workload's neuron keep, over several layers' weights
    in turn (so that every launch reads from HBM)."""
    import numpy as np
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    dvbuild.build()
    dv.lib()
    w = workload(a)
    L = min(w.layers, 6)
    kN = traffic.k_of(w.keep_N, w.F)
    D = dv.dims(w.d, w.h, w.h_kv, w.dh, w.F, w.r, 8)
    ws = dv.workspace(D, w.B)
    x = synth.hidden(w, device=dev)
    out = torch.empty(w.B, w.d, dtype=torch.float16, device=dev)
    layers = []
    for l in range(L):
        W = synth.layer_weights(w, l, device=dev)
        W = {k: W[k] for k in ("fc1", "fc2T", "b1", "ln2_g", "ln2_b") if k in W}
        idx = np.sort(np.random.default_rng(l).choice(w.F, kN, replace=False)).astype(np.int32)
        layers.append((W, dv.quantize_w4(W["fc1"]), dv.quantize_w4(W["fc2T"]),
                       torch.from_numpy(idx).to(dev)))
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    stream = torch.cuda.Stream(device=dev)
    res = {}
    for name in ("fp16", "w4"):
        def one(l):
            W, q1, q2, idx = layers[l % L]
            if name == "fp16":
                dv.sparse_mlp(x, D, W, idx, kN, out, ws, stream=stream)
            else:
                dv.sparse_mlp_w4(x, D, W, q1, q2, idx, kN, out, ws, stream=stream)
        with torch.cuda.stream(stream):
            for l in range(max(3, a.warmup) * L):
                one(l)
        torch.cuda.synchronize()
        reps = max(L, (a.steps // L) * L)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for l in range(reps):
                one(l)
            e1.record(stream)
        torch.cuda.synchronize()
        # the streaming kernel alone, event-bracketed
        prof = dv.Profiler(cap=8 * L + 16)
        with torch.cuda.stream(stream):
            prof.start()
            for l in range(L):
                one(l)
            prof.stop()
        torch.cuda.synchronize()
        ks = [ms * 1e3 for tag, ms in prof.durations_ms() if tag == "mlp"]
        res[name] = {"us_per_block": e0.elapsed_time(e1) * 1e3 / reps,
                     "kernel_us": sum(ks) / len(ks)}
    pk, pk_src = peaks()
    row = {"fp16": 2 * w.d, "w4": dv.w4_row_bytes(w.d)}
    out_j = {"metric": "mlp_block_w4a16", "workload": workload_name(w), "data": "synthetic",
             "neurons": kN, "layers_rotated": L}
    for name in ("fp16", "w4"):
        by = 2 * kN * row[name]
        kus = res[name]["kernel_us"]
        out_j[name] = {"us_per_block": round(res[name]["us_per_block"], 2),
                       "stream_kernel_us": round(kus, 2), "weight_bytes": by,
                       "gbs": round(by / kus / 1e3, 1),
                       "frac": round(by / kus / 1e3 / pk, 3), "peak_gbs": pk,
                       "peak_source": pk_src}
    out_j["speedup"] = round(res["fp16"]["us_per_block"] / res["w4"]["us_per_block"], 3)
    print(json.dumps(out_j))


def run_gate(a):
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    dvbuild.build()
    dv.lib()
    base = workload(a)
    cal = [int(x) for x in a.gate_ctx.split(",")]
    val = [int(x) for x in a.gate_val.split(",")]
    every = sorted(set(cal) | set(val) | {c for c, _, _ in GATE_MIX})
    steps = max(5, min(a.steps, 50))
    T = {m: {} for m in range(4)}
    S = {}
    for n in every:
        for m in range(4):
            kn, kh, kkv = GATE_KEEP[m](base)
            w = dataclasses.replace(base, n=n, keep_N=kn, keep_H=kh, keep_KV=kkv)
            T[m][n], sel = _time_mode(w, dev, steps, a.warmup)
            if sel:
                S.setdefault(n, []).append(sel)
        print(f"[gate] n {n}: " + ", ".join(f"{dv.MODES[m]} {T[m][n]:.1f}" for m in range(4))
              + f" us/layer, scoring {statistics.mean(S[n]):.0f} us/layer", file=sys.stderr, flush=True)
    sel_us = {n: float(statistics.mean(v)) for n, v in S.items()}
    D = dv.dims(base.d, base.h, base.h_kv, base.dh, base.F, base.r, 1)
    keep = dv.Keep(base.keep_N, base.keep_H, base.keep_KV)
    cm = dv.cost_calibrate(D, keep, dv.request(), [float(c) for c in cal],
                           [[T[m][c] for c in cal] for m in range(4)], [sel_us[c] for c in cal])
    per_step = dv.request(steps=10**9)   # per-step times, the scoring pass left out
    checks = []
    for n in val:
        p = dv.plan_decode(D, keep, per_step, cm, float(n))
        checks.append({"n": n, "measured_us": [round(T[m][n], 2) for m in range(4)],
                       "predicted_us": [round(x, 2) for x in p["us"]],
                       "err_pct": [round(100 * (p["us"][m] / T[m][n] - 1), 2) for m in range(4)]})
    pairs = [(dv.MODE_DENSE, dv.MODE_ACT), (dv.MODE_DENSE, dv.MODE_KV),
             (dv.MODE_ACT, dv.MODE_KV), (dv.MODE_ACT, dv.MODE_COMPOSED),
             (dv.MODE_KV, dv.MODE_COMPOSED), (dv.MODE_DENSE, dv.MODE_COMPOSED)]
    crossings = []
    for x, y in pairs:
        pred = dv.plan_crossing(D, keep, per_step, cm, x, y, float(every[0]), float(every[-1]))
        meas = _measured_crossing(every, [T[x][n] for n in every], [T[y][n] for n in every])
        crossings.append({"modes": f"{dv.MODES[x]}/{dv.MODES[y]}",
                          "predicted": None if pred is None else round(pred),
                          "measured": None if meas is None else round(meas)})
    # dispatch: each request runs its decode steps in one mode, paying the
    # scoring pass once if that mode selects KV
    def cost(mode, n, st):
        return st * T[mode][n] + (sel_us[n] if mode in (dv.MODE_KV, dv.MODE_COMPOSED) else 0.0)
    totals = {name: 0.0 for name in list(dv.MODES) + ["gate"]}
    picks = []
    for n, st, count in GATE_MIX:
        choice = dv.plan_decode(D, keep, dv.request(steps=st), cm, float(n))["choice"]
        picks.append({"n": n, "steps": st, "mode": dv.MODES[choice]})
        for mode in range(4):
            totals[dv.MODES[mode]] += count * cost(mode, n, st)
        totals["gate"] += count * cost(choice, n, st)
    best = sum(count * min(cost(mode, n, st) for mode in range(4))
                      for n, st, count in GATE_MIX)
    speedup = {k: round(totals["dense"] / v, 3) for k, v in totals.items()}
    out = {
        "metric": "latency_gate", "workload": workload_name(base), "data": "synthetic",
        "calibration_ctx": cal, "validation_ctx": val, "steps_timed": steps,
        "us_per_layer": {dv.MODES[m]: {str(n): round(T[m][n], 2) for n in every} for m in range(4)},
        "scoring_us_per_layer": {str(n): round(v, 1) for n, v in sel_us.items()},
        "cost_us": {dv.MODES[m]: [round(cm.cost_us[m][i], 2) for i in range(len(cal))]
                    for m in range(4)},
        "validation": checks, "crossings": crossings, "dispatch": picks,
        "mix_speedup_over_dense": speedup,
        "mix_gate_vs_best_per_request": round(best / totals["gate"], 4),
    }
    print(json.dumps(out))


def main():
    a = parse()
    if a.impl == "reference":
        run_reference(a)
    elif a.gate:
        run_gate(a)
    elif a.decode_steps:
        run_multistep(a)
    elif a.union_tc:
        run_union_tc(a)
    elif a.w4 and a.step:
        run_w4_step(a)
    elif a.w4:
        run_w4(a)
    else:
        run_ours(a)


if __name__ == "__main__":
    main()
