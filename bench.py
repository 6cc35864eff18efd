"""Benchmark of the QSA layer hot path on GB300.

One step = 12 QSA layers (distinct, seeded synthetic buffers per layer) of each of:
  A  prefill  T=1984 at pos0=0      (identity: every causal cell)       qsa_flash_prefill
  B  prefill  T=1984 at pos0=30000  (31,984-cell cache, top-2048)       qsa_select + qsa_flash_prefill
  C  decode   N=1 at P=8192         (top-2048)                          qsa_decode_layer (select, attend, merge:
                                                                          one launch)
value = identity-prefill tokens per second per layer (T=1984, the pages' own convention: tokens of
the window / time of one layer), from the A part of the timed steps, times the number of replicas.
The timed steps replay one CUDA graph per workload (captured from the same API calls); --eager
times the calls themselves.  After the timed steps, every configuration of the workload list is
timed on its own (CUDA graphs of the API calls, L2 flushed before each replay) and reported under
"configs" with the per-call roofline fractions.

python bench.py [--gpus N --steps K --warmup W] [--impl reference]
Under torchrun (N > 1) every rank runs the same step on its own GPU (replicas, weak scaling)
and rank 0 prints one JSON line with the max step time over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

LAYERS = 12
T_PREFILL = 1984
POS0_B = 30000
N_DEC, P_DEC = 1, 8192
HEADS, D = 24, 256
METRIC = "prefill tokens/s per QSA layer (T=1984) + decode us/token; % tensor/HBM roofline"
UNIT = "tokens/s per layer (identity prefill T=1984)"


def flops_prefill(T, pos0, topk=2048, idmax=2051):
    """Algorithmic FLOPs of one prefill layer: 24 heads x cells attended x 256 x (2 for QK + 2 for PV)."""
    cells = 0
    for t in range(T):
        n = pos0 + t + 1
        cells += n if n <= idmax else topk
    return 24 * cells * 256 * 4


KERNEL_OF_FAMILY = {"dense_prefill": "flash_dense_kernel", "gather_prefill": "flash_gather_kernel"}


def recorded_traffic(kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu record, or None when the
    kernel's source has changed since the counters were taken."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)[kernel]
        with open(os.path.join(ROOT, rec["source"]), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != rec["source_sha256"]:
                return None
        return rec["dram_bytes_per_launch"]
    except Exception:
        return None


def max_over_ranks(x, dist, device):
    """The slowest rank's time: every rank contributes x, every rank gets the maximum."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(ms_per_layer_set, world):
    """Identity-prefill tokens/s per layer of the whole job: each of `world` replicas runs the 12
    identity-prefill layers of T=1984 tokens in ms_per_layer_set (the max over ranks)."""
    return T_PREFILL / (ms_per_layer_set * 1e-3 / LAYERS) * world


def read_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], p.get("bf16_tflops_sustained", p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    def __init__(self, index, path, keep=True):
        self.path = path
        self.keep = keep  # False: the CSV is a temporary file, removed once read
        self.proc = None
        self.f = None
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.f = open(path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(index), f"--query-gpu={q}", "--format=csv,noheader",
                                          "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:  # no nvidia-smi: no clock record
            self.proc = None
            if self.f:
                self.f.close()
            self._discard()

    def _discard(self):
        if not self.keep:
            try:
                os.remove(self.path)
            except OSError:
                pass

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        try:
            return self._summary()
        finally:
            self._discard()

    def _summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1].split()[0]))
                mx.append(float(parts[2].split()[0]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons), "samples": len(sm)}


def make_layers(device, torch, synth):
    """Seeded synthetic buffers for the 12 layers of each workload (seed 5 + layer)."""
    A, B, C = [], [], []
    for l in range(LAYERS):
        inp = synth.layer_inputs(T_PREFILL, T_PREFILL, seed=5 + l)
        A.append({k: torch.from_numpy(v).to(device) for k, v in inp.items()})
        inp = synth.layer_inputs(T_PREFILL, POS0_B + T_PREFILL, seed=105 + l)
        B.append({k: torch.from_numpy(v).to(device) for k, v in inp.items()})
        inp = synth.layer_inputs(N_DEC, P_DEC + N_DEC, seed=205 + l)
        C.append({k: torch.from_numpy(v).to(device) for k, v in inp.items()})
    return A, B, C


def run_ours(args, rank, world, local_rank):
    import torch

    from int8_kv_top_gb300 import qsa, synth

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    qsa.load()
    A, B, C = make_layers(device, torch, synth)
    nA, nB, nC = T_PREFILL, POS0_B + T_PREFILL, P_DEC + N_DEC
    cap = qsa.chunk_cap_for()
    outA = [torch.empty((T_PREFILL, HEADS, D), dtype=torch.float16, device=device) for _ in range(LAYERS)]
    outB = [torch.empty((T_PREFILL, HEADS, D), dtype=torch.float16, device=device) for _ in range(LAYERS)]
    idsB = [torch.empty((T_PREFILL, 2, 2048), dtype=torch.int32, device=device) for _ in range(LAYERS)]
    idsC = [torch.empty((N_DEC, 2, 2048), dtype=torch.int32, device=device) for _ in range(LAYERS)]
    partC = torch.empty((N_DEC, cap, HEADS, 258), device=device)
    nchC = torch.empty(N_DEC, dtype=torch.int32, device=device)
    xpC = [torch.empty((N_DEC, HEADS, D), device=device) for _ in range(LAYERS)]
    wsB = torch.empty(qsa.qsa_select_workspace_bytes(T_PREFILL, POS0_B, nB), dtype=torch.uint8, device=device)
    wsC = torch.empty(qsa.qsa_select_workspace_bytes(N_DEC, P_DEC, nC), dtype=torch.uint8, device=device)
    pwsB = torch.empty(qsa.qsa_flash_prefill_workspace_bytes(T_PREFILL, POS0_B, nB), dtype=torch.uint8, device=device)
    pwsA = torch.empty(qsa.qsa_flash_prefill_workspace_bytes(T_PREFILL, 0, nA), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    # our kernel launches per step (the select workspace memset is not counted):
    # A mirror 1 + dense 1; B select 4 (prep_q, prep_k, score, top-k) + mirror 1 + gather 1;
    # C select 2 (score_small, top-k) + partial 1 + merge 1
    launches_per_step = LAYERS * (2 + 6 + 1)

    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def mark_in(marks):
        def mark(name):
            if marks is not None:
                e = ev()
                e.record(stream)
                marks.append((name, e))
        return mark

    def sec_a(marks=None):
        mark = mark_in(marks)
        mark("A0")
        for l in range(LAYERS):
            d = A[l]
            qsa.qsa_flash_prefill(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], nA, T_PREFILL, 0, None, outA[l], pwsA)
        mark("A1")

    def sec_b(marks=None):
        mark = mark_in(marks)
        for l in range(LAYERS):
            d = B[l]
            mark("Bs")
            qsa.qsa_select(d["q"], d["kq"], d["ksc"], nB, T_PREFILL, POS0_B, idsB[l], wsB)
            mark("Bf")
            qsa.qsa_flash_prefill(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], nB, T_PREFILL, POS0_B, idsB[l],
                                  outB[l], pwsB)
        mark("C0")

    def sec_c(marks=None):
        mark = mark_in(marks)
        for l in range(LAYERS):
            d = C[l]
            mark("Cs")
            qsa.qsa_decode_layer(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], nC, N_DEC, P_DEC, idsC[l], xpC[l])
        mark("C1")

    def step(marks=None):
        sec_a(marks)
        sec_b(marks)
        sec_c(marks)

    for _ in range(args.warmup):
        step()
    qsa.qsa_check_device_status()

    # The timed steps replay one CUDA graph per workload (the same kernels on the same resident
    # buffers, without the per-call host work); eager steps with events between the calls give
    # the per-kernel-family breakdown afterwards.
    graphs = None
    if not args.eager:
        try:
            graphs = []
            for sec in (sec_a, sec_b, sec_c):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    sec()
                graphs.append(g)
            for g in graphs:
                g.replay()
            torch.cuda.synchronize(device)
            qsa.qsa_check_device_status()
        except Exception as exc:  # capture not available: time the eager calls instead
            print(f"graph capture failed ({exc}); timing eager calls", file=sys.stderr)
            graphs = None

    dist = None
    if world > 1:
        import torch.distributed as dist
    # ---- timed region: K steps, barrier + sync on both sides
    # nvidia-smi samples of the timed region go to --clocks-csv if given, else to a temporary file
    clocks_path = args.clocks_csv.replace("{rank}", str(rank)) if args.clocks_csv else \
        os.path.join(tempfile.gettempdir(), f"qsa_bench_clocks_rank{rank}_{os.getpid()}.csv")
    sampler = ClockSampler(local_rank, clocks_path, keep=bool(args.clocks_csv))
    all_marks = []
    sec_ms = [0.0, 0.0, 0.0]
    if dist:
        dist.barrier()
    torch.cuda.synchronize(device)
    e0, e1 = ev(), ev()
    e0.record(stream)
    sec_events = []
    for _ in range(args.steps):
        if graphs:
            evs = [ev() for _ in range(4)]
            for i, g in enumerate(graphs):
                evs[i].record(stream)
                g.replay()
            evs[3].record(stream)
            sec_events.append(evs)
        else:
            marks = []
            step(marks)
            all_marks.append(marks)
    e1.record(stream)
    torch.cuda.synchronize(device)
    for evs in sec_events:
        for i in range(3):
            sec_ms[i] += evs[i].elapsed_time(evs[i + 1]) / args.steps
    if dist:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    qsa.qsa_check_device_status()
    total_ms = e0.elapsed_time(e1)
    total_ms = max_over_ranks(total_ms, dist, device)
    ms_step = total_ms / args.steps

    if graphs:  # eager marked steps for the per-kernel-family breakdown (outside the timed region)
        for _ in range(min(args.steps, 5)):
            marks = []
            step(marks)
            all_marks.append(marks)
        torch.cuda.synchronize(device)
        qsa.qsa_check_device_status()

    # ---- per-kernel-family times from the marks (averaged over steps)
    fam = {"dense_prefill": 0.0, "select_B": 0.0, "gather_prefill": 0.0, "decode_layer": 0.0}
    for marks in all_marks:
        names = [m[0] for m in marks]
        evs = [m[1] for m in marks]
        for i, n in enumerate(names[:-1]):
            dt = evs[i].elapsed_time(evs[i + 1])
            nxt = names[i + 1]
            if n == "A0":
                fam["dense_prefill"] += dt
            elif n == "Bs":
                fam["select_B"] += dt
            elif n == "Bf":
                fam["gather_prefill"] += dt
            elif n == "Cs":
                fam["decode_layer"] += dt
            del nxt
    fam = {k: v / max(1, len(all_marks)) for k, v in fam.items()}  # ms per step (12 launches each)
    # per-workload times of the timed steps: graph replays when available, else the eager marks
    if graphs:
        sec = {"A": sec_ms[0], "B": sec_ms[1], "C": sec_ms[2]}
    else:
        sec = {"A": fam["dense_prefill"], "B": fam["select_B"] + fam["gather_prefill"],
               "C": fam["decode_layer"]}

    # ---- e2e: same step through the public API from pinned host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, torch, qsa, device, stream, A, B, C, outA, outB, idsB, idsC, partC, nchC, xpC, wsB, wsC,
                      pwsA, pwsB, nA, nB, nC, cap, dist)

    hbm_gbs, bf16_tf, bf16_tf_sus, peak_src = read_peaks()
    flopA = flops_prefill(T_PREFILL, 0)
    flopB = flops_prefill(T_PREFILL, POS0_B)
    # kernels are timed inside steps of about a millisecond or less: the burst peaks apply
    per_launch = {
        "dense_prefill": {"bound": "tensor", "achieved": flopA / (sec["A"] / LAYERS * 1e-3) / 1e12,
                          "peak": bf16_tf, "unit": "TFLOP/s",
                          "call": "qsa_flash_prefill T=1984 pos0=0 (fp16 mirror + flash_dense_kernel), graph-timed"},
        "gather_prefill": {"bound": "tensor", "achieved": flopB / (fam["gather_prefill"] / LAYERS * 1e-3) / 1e12,
                           "peak": bf16_tf, "unit": "TFLOP/s",
                           "call": "qsa_flash_prefill T=1984 pos0=30000 (fp16 mirror + flash_gather_kernel), eager",
                           # the selected rows are gathered from L2: T x 2 groups x 2048 cells x 1 KB (K^ + V^ fp16)
                           "l2_gather_gbs": T_PREFILL * 2 * 2048 * 1024 / (fam["gather_prefill"] / LAYERS * 1e-3) / 1e9},
    }
    for v in per_launch.values():
        v["frac"] = v["achieved"] / v["peak"]
    for k, v in per_launch.items():
        v["traffic"] = recorded_traffic(KERNEL_OF_FAMILY[k])
    dominant = max(("dense_prefill", "gather_prefill"), key=lambda k: fam[k])
    roof = dict(per_launch[dominant])
    roof["kernel"] = KERNEL_OF_FAMILY[dominant]
    roof["traffic_unit"] = "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)"
    roof["peak_source"] = f"{peak_src}, burst bf16 (f16 same rate)"

    configs = None
    if not args.no_configs:
        configs = measure_configs(torch, qsa, synth, device, stream, (hbm_gbs, bf16_tf), A, B)
        for k in ("select_prefill", "decode_select", "decode_partial", "merge", "decode_layer", "decode_layer_batched",
                  "prep"):
            if k in configs.get("hbm_calls", {}):
                per_launch[k] = configs["hbm_calls"][k]
        if "prefill_batched" in configs:
            per_launch["prefill_batched"] = dict(configs["prefill_batched"]["hbm"],
                                                 call="qsa_flash_prefill_batched 64 x T=128")

    value = whole_job_rate(max_over_ranks(sec["A"], dist, device), world)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16 operands, f32 accumulate", "data": "synthetic (seeded; q~N(0,1) fp16, int8 K/V uniform "
        "[-127,127], fp16 scales U[0.005,0.02])",
        "config": {"workload": "prefill T=1984 pos0=0, 12 QSA layers (identity ids; the value); each timed step "
                               "also runs 12 layers of prefill T=1984 pos0=30000 (31984-cell cache, top-2048) and "
                               "12 layers of decode N=1 P=8192 (qsa_decode_layer)", "layers": LAYERS,
                   "heads": "2 KV x 12 q, dim 256", "l2": "inputs larger than L2 (12 distinct layer buffer sets)",
                   "parallelism": f"replicas x{world}"},
        "value_definition": "T / (time of one identity-prefill layer), T = 1984, times replicas",
        "breakdown_ms_per_step": fam,
        "breakdown_timing": "eager calls, CUDA events between them",
        "timing": "CUDA graph replay per workload" if graphs else "eager calls",
        "workload_ms_per_step": sec,
        "prefill_identity_us_per_layer": sec["A"] / LAYERS * 1e3,
        "prefill_selected_us_per_layer": sec["B"] / LAYERS * 1e3,
        "decode_us_per_token_per_layer": sec["C"] / LAYERS * 1e3 / N_DEC,
        "roofline": roof, "roofline_per_kernel": per_launch,
        "configs": configs,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks, "e2e": e2e,
    }
    return line


def _graph_us(torch, device, stream, fn, reps, flush):
    """fn() captured in one CUDA graph, replayed `reps` times, each replay after an L2 flush (a
    256 MB write) outside the timed events.  Returns (median, min) replay time in microseconds."""
    fn()
    torch.cuda.synchronize(device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    g.replay()
    torch.cuda.synchronize(device)
    evs = []
    for _ in range(reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize(device)
    us = sorted(a.elapsed_time(b) * 1e3 for a, b in evs)
    del g
    return statistics.median(us), us[0]


def _roof(achieved, peak, unit, bound):
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak}


def measure_configs(torch, qsa, synth, device, stream, peaks, A, B, reps=10):
    """Every configuration of the workload list timed on its own, with the per-call roofline.

    0: prefill T=96 pos0=0, 1 layer; 1: T=512 pos0=0, 12 layers; 2: T=1984 pos0=0, 12 layers;
    3: T=1984 pos0=30000 over 31,984 cells, select and prefill, 12 layers; 4: decode N in {1, 4} x
    P in {512, 2048, 8192}, select / partial / merge and their total, 12 layers.  Tensor fractions
    count only causal or selected cells; HBM fractions count the bytes the method must move, each
    needed cell once per call (distinct (cell, group) rows, from the ids the call produced)."""
    hbm_gbs, tf_burst = peaks
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    res = {"timing": "CUDA graph of the API calls over 12 distinct layer buffer sets (1 for config 0); median of "
                     f"{reps} replays, L2 flushed (256 MB write) before each replay outside the timed events",
           "peaks": {"hbm_gbs": hbm_gbs, "bf16_tflops_burst": tf_burst}}
    gt = lambda fn: _graph_us(torch, device, stream, fn, reps, flush)  # noqa: E731
    up = lambda inp: {k: torch.from_numpy(v).to(device) for k, v in inp.items()}  # noqa: E731

    def prefill_set(T, pos0, bufs, ids=None):
        n = pos0 + T
        outs = [torch.empty((T, HEADS, D), dtype=torch.float16, device=device) for _ in bufs]
        ws = torch.empty(qsa.qsa_flash_prefill_workspace_bytes(T, pos0, n), dtype=torch.uint8, device=device)

        def fn():
            for l, d in enumerate(bufs):
                qsa.qsa_flash_prefill(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], n, T, pos0,
                                      None if ids is None else ids[l], outs[l], ws)
        return fn

    def prefill_entry(T, pos0, layers, med, mn):
        fl = flops_prefill(T, pos0)
        per_layer = med / layers
        return {"T": T, "pos0": pos0, "layers": layers, "us_per_layer": per_layer, "us_per_layer_min": mn / layers,
                "ms_per_layers": med * 1e-3, "tokens_per_s_per_layer": T / (per_layer * 1e-6),
                "gflop_per_layer": fl / 1e9,
                "tensor": _roof(fl / (per_layer * 1e-6) / 1e12, tf_burst, "TFLOP/s", "tensor")}

    # configs 0-2: identity prefill
    b0 = [up(synth.layer_inputs(96, 96, seed=5))]
    res["config0"] = prefill_entry(96, 0, 1, *gt(prefill_set(96, 0, b0)))
    b1 = [up(synth.layer_inputs(512, 512, seed=5 + l)) for l in range(LAYERS)]
    res["config1"] = prefill_entry(512, 0, LAYERS, *gt(prefill_set(512, 0, b1)))
    res["config2"] = prefill_entry(T_PREFILL, 0, LAYERS, *gt(prefill_set(T_PREFILL, 0, A)))
    # the same layers with the output gate applied in the epilogue (qsa_flash_prefill_gated)
    gates = [torch.from_numpy(synth.gate_input(T_PREFILL, seed=500 + l)).to(device) for l in range(LAYERS)]
    outg = [torch.empty((T_PREFILL, HEADS, D), dtype=torch.float16, device=device) for _ in range(LAYERS)]
    wsg = torch.empty(qsa.qsa_flash_prefill_workspace_bytes(T_PREFILL, 0, T_PREFILL), dtype=torch.uint8, device=device)

    def gated2():
        for l, d in enumerate(A):
            qsa.qsa_flash_prefill_gated(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], T_PREFILL, T_PREFILL, 0, None,
                                        gates[l], outg[l], wsg)
    res["config2_gated"] = prefill_entry(T_PREFILL, 0, LAYERS, *gt(gated2))
    del b0, b1, gates, outg, wsg

    # the fused prep of the same windows (T=1984 new tokens; norm + rotary + quantise into the cache)
    preps = [{k: torch.from_numpy(v).to(device) for k, v in synth.prep_inputs(T_PREFILL, seed=700 + l).items()}
             for l in range(LAYERS)]
    qcur = [torch.empty((T_PREFILL, HEADS, D), dtype=torch.float16, device=device) for _ in range(LAYERS)]

    def prep_all():
        for l, d in enumerate(A):
            pi = preps[l]
            qsa.qsa_prep(pi["q_raw"], pi["k_raw"], pi["v_raw"], pi["q_gamma"], pi["k_gamma"], T_PREFILL, 0, T_PREFILL,
                         qcur[l], None, d["kq"], d["ksc"], d["vq"], d["vsc"])
    med, mn = gt(prep_all)
    per_layer = med / LAYERS
    by = T_PREFILL * ((HEADS + 4) * D * 2 + HEADS * D * 2 + 2 * 2 * (D + 8))
    res["prep"] = {"T": T_PREFILL, "us_per_layer": per_layer, "tokens_per_s_per_layer": T_PREFILL / (per_layer * 1e-6),
                   "bytes": by, "bytes_note": "raw q, k, v rows read; qcur, the int8 K/V rows and scales written",
                   "hbm": _roof(by / (per_layer * 1e-6) / 1e9, hbm_gbs, "GB/s", "hbm"), "call": "qsa_prep"}
    del preps, qcur

    # config 3: select, then the gathered prefill, and both
    nB = POS0_B + T_PREFILL
    idsB = [torch.empty((T_PREFILL, 2, 2048), dtype=torch.int32, device=device) for _ in range(LAYERS)]
    wsB = torch.empty(qsa.qsa_select_workspace_bytes(T_PREFILL, POS0_B, nB), dtype=torch.uint8, device=device)

    def sel3():
        for l, d in enumerate(B):
            qsa.qsa_select(d["q"], d["kq"], d["ksc"], nB, T_PREFILL, POS0_B, idsB[l], wsB)
    fl3 = prefill_set(T_PREFILL, POS0_B, B, idsB)
    s_med, s_min = gt(sel3)
    f_med, f_min = gt(fl3)
    b_med, b_min = gt(lambda: (sel3(), fl3()))
    e3 = prefill_entry(T_PREFILL, POS0_B, LAYERS, b_med, b_min)
    e3["n_cells"] = nB
    sel_bytes = nB * 2 * 264 + T_PREFILL * HEADS * D * 2 + T_PREFILL * 2 * 2048 * 4
    e3["select_us_per_layer"] = s_med / LAYERS
    e3["select_hbm"] = _roof(sel_bytes / (s_med / LAYERS * 1e-6) / 1e9, hbm_gbs, "GB/s", "hbm")
    e3["select_hbm"]["bytes"] = sel_bytes
    e3["select_hbm"]["bytes_note"] = ("K codes and scales of every cell (both groups), q, ids; the fp16 score "
                                      "matrix this implementation writes and reads back is not counted")
    e3["select_tensor"] = _roof(2 * 2 * (POS0_B * T_PREFILL + T_PREFILL * (T_PREFILL + 1) // 2) * 256
                                / (s_med / LAYERS * 1e-6) / 1e12, tf_burst, "TFLOP/s", "tensor")
    e3["select_tensor"]["flop_note"] = "Qsum form: 2 x 256 per (token, group, causal cell)"
    e3["flash_us_per_layer"] = f_med / LAYERS
    e3["flash_tensor"] = _roof(flops_prefill(T_PREFILL, POS0_B) / (f_med / LAYERS * 1e-6) / 1e12, tf_burst,
                               "TFLOP/s", "tensor")
    res["config3"] = e3
    hbm_calls = {"select_prefill": dict(e3["select_hbm"], call="qsa_select T=1984 pos0=30000"),
                 "prep": dict(res["prep"]["hbm"], call="qsa_prep T=1984")}

    # config 4: decode
    cap = qsa.chunk_cap_for()
    dec = {}
    for N in (1, 4):
        for P in (512, 2048, 8192):
            n = P + N
            bufs = [up(synth.layer_inputs(N, n, seed=2000 + 10 * N + P + l)) for l in range(LAYERS)]
            ids = [torch.full((N, 2, 2048), -1, dtype=torch.int32, device=device) for _ in range(LAYERS)]
            part = [torch.empty((N, cap, HEADS, 258), device=device) for _ in range(LAYERS)]
            nch = [torch.empty(N, dtype=torch.int32, device=device) for _ in range(LAYERS)]
            xp = [torch.empty((N, HEADS, D), device=device) for _ in range(LAYERS)]
            wsz = qsa.qsa_select_workspace_bytes(N, P, n)
            ws = torch.empty(max(wsz, 16), dtype=torch.uint8, device=device)
            any_sel = n > 2051

            def fsel():
                for l, d in enumerate(bufs):
                    qsa.qsa_select(d["q"], d["kq"], d["ksc"], n, N, P, ids[l], ws)

            def fpart():
                for l, d in enumerate(bufs):
                    qsa.qsa_decode_partial(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], n, N, P,
                                           ids[l] if any_sel else None, part[l], nch[l], cap)

            def fmerge():
                for l in range(LAYERS):
                    qsa.qsa_merge(part[l], nch[l], N, cap, xp[l])
            fsel()
            fpart()
            torch.cuda.synchronize(device)
            qsa.qsa_check_device_status()
            # distinct (cell, group) rows each call must read, and the partial chunks it writes
            ids0 = ids[0].cpu().numpy()
            rows, chunks = 0, 0
            for g in range(2):
                cells = set()
                for t in range(N):
                    n_kv = P + t + 1
                    if n_kv <= 2051:
                        cells.update(range(n_kv))
                        chunks += (n_kv + 63) // 64 if g == 0 else 0
                    else:
                        cells.update(int(c) for c in ids0[t, g])
                        chunks += 2048 // 64 if g == 0 else 0
                rows += len(cells)
            n_sel_tok = sum(1 for t in range(N) if P + t + 1 > 2051)
            by_sel = n * 2 * 264 + N * HEADS * D * 2 + n_sel_tok * 2 * 2048 * 4 if any_sel else 0
            by_part = rows * 528 + N * HEADS * D * 2 + chunks * HEADS * 258 * 4
            by_merge = chunks * HEADS * 258 * 4 + N * HEADS * D * 4
            e = {"N": N, "P": P}
            for name, fn, by in (("select", fsel, by_sel), ("partial", fpart, by_part), ("merge", fmerge, by_merge)):
                if name == "select" and not any_sel:
                    e[name] = {"us_per_call": 0.0, "note": "no token above the identity threshold: nothing launched"}
                    continue
                med, _ = gt(fn)
                per_call = med / LAYERS
                e[name] = {"us_per_call": per_call, "us_per_token": per_call / N, "bytes": by,
                           "hbm": _roof(by / (per_call * 1e-6) / 1e9, hbm_gbs, "GB/s", "hbm")}
            med, _ = gt(lambda: (fsel() if any_sel else None, fpart(), fmerge()))
            # the layer as a whole: K of every cell once (selection), V of the selected rows (K and V of
            # every cell when no token selects), q, the merged output and the ids
            kv_bytes = n * 2 * 264 + rows * 264 if any_sel else rows * 528
            tot_bytes = kv_bytes + N * HEADS * D * 2 + N * HEADS * D * 4 + n_sel_tok * 2 * 2048 * 4
            e["total"] = {"us_per_call": med / LAYERS, "us_per_token_per_layer": med / LAYERS / N,
                          "bytes": tot_bytes, "bytes_note": "each needed input row read once, the merged output "
                          "and the ids written once (partials between the calls not counted)",
                          "hbm": _roof(tot_bytes / (med / LAYERS * 1e-6) / 1e9, hbm_gbs, "GB/s", "hbm")}
            # the same step in one launch (qsa_decode_layer): select, attend and merge fused
            xpf = [torch.empty((N, HEADS, D), device=device) for _ in range(LAYERS)]
            idf = [torch.empty((N, 2, 2048), dtype=torch.int32, device=device) for _ in range(LAYERS)]

            def ffused():
                for l, d in enumerate(bufs):
                    qsa.qsa_decode_layer(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], n, N, P, idf[l], xpf[l])
            med, _ = gt(ffused)
            e["fused"] = {"us_per_call": med / LAYERS, "us_per_token_per_layer": med / LAYERS / N,
                          "bytes": tot_bytes, "launches": 1,
                          "hbm": _roof(tot_bytes / (med / LAYERS * 1e-6) / 1e9, hbm_gbs, "GB/s", "hbm")}
            dec[f"N{N}_P{P}"] = e
            if N == 1 and P == 8192:
                for k, name in (("decode_select", "select"), ("decode_partial", "partial"), ("merge", "merge"),
                                ("decode_layer", "fused")):
                    hbm_calls[k] = dict(e[name]["hbm"], call=f"{name} N=1 P=8192", us_per_call=e[name]["us_per_call"])
            del bufs, ids, part, nch, xp, ws, xpf, idf
    res["config4_decode"] = dec
    # continuous batching: 64 sequences of one decode token each at P=8192 in one launch
    B_SEQ, P_B = 64, 8192
    n1 = P_B + 1
    pool = {}
    parts = [synth.layer_inputs(1, n1, seed=3000 + b) for b in range(B_SEQ)]
    for k in ("q", "kq", "vq", "ksc", "vsc"):
        pool[k] = torch.from_numpy(np.concatenate([pc[k] for pc in parts], axis=0)).to(device)
    del parts
    seqs = torch.tensor([[b * n1, n1, P_B, b] for b in range(B_SEQ)], dtype=torch.int32, device=device)
    ids_b = torch.empty((B_SEQ, 2, 2048), dtype=torch.int32, device=device)
    xp_b = torch.empty((B_SEQ, HEADS, D), device=device)

    def fbatch():
        qsa.qsa_decode_layer_batched(pool["q"], pool["kq"], pool["vq"], pool["ksc"], pool["vsc"], B_SEQ * n1, seqs,
                                     B_SEQ, B_SEQ, n1, ids_b, xp_b)
    med, mn = gt(fbatch)
    fbatch()
    torch.cuda.synchronize(device)
    qsa.qsa_check_device_status()
    idn = ids_b.cpu().numpy()
    rows = sum(len(np.unique(idn[b, g])) for b in range(B_SEQ) for g in range(2))
    by = B_SEQ * n1 * 2 * 264 + rows * 264 + B_SEQ * HEADS * D * (2 + 4) + B_SEQ * 2 * 2048 * 4
    res["decode_batched"] = {"sequences": B_SEQ, "tokens_per_sequence": 1, "P": P_B, "us_per_launch": med,
                             "us_per_launch_min": mn, "tokens_per_s": B_SEQ / (med * 1e-6), "bytes": by,
                             "hbm": _roof(by / (med * 1e-6) / 1e9, hbm_gbs, "GB/s", "hbm"),
                             "call": "qsa_decode_layer_batched, one launch"}
    hbm_calls["decode_layer_batched"] = dict(res["decode_batched"]["hbm"], call="qsa_decode_layer_batched 64 x P=8192")
    del pool
    # continuous batching of prompts: 64 sequences of 128 new tokens each (no cached prefix) in one
    # batched prefill call, against the same 64 prompts as 64 single-sequence calls
    P_SEQ, P_T = 64, 128
    parts = [synth.layer_inputs(P_T, P_T, seed=3500 + b) for b in range(P_SEQ)]
    pool = {k: torch.from_numpy(np.concatenate([pc[k] for pc in parts], axis=0)).to(device)
            for k in ("q", "kq", "vq", "ksc", "vsc")}
    singles = [up(pc) for pc in parts]
    del parts
    seqs = torch.tensor([[b * P_T, P_T, 0, b * P_T] for b in range(P_SEQ)], dtype=torch.int32, device=device)
    n_tok = P_SEQ * P_T
    out_p = torch.empty((n_tok, HEADS, D), dtype=torch.float16, device=device)
    ws_p = torch.empty(qsa.qsa_flash_prefill_batched_workspace_bytes(P_SEQ, n_tok, P_T), dtype=torch.uint8,
                       device=device)

    def fpb():
        qsa.qsa_flash_prefill_batched(pool["q"], pool["kq"], pool["vq"], pool["ksc"], pool["vsc"], n_tok, seqs, P_SEQ,
                                      n_tok, P_T, None, out_p, ws_p)
    med, mn = gt(fpb)
    outs1 = [torch.empty((P_T, HEADS, D), dtype=torch.float16, device=device) for _ in range(P_SEQ)]
    ws1 = torch.empty(qsa.qsa_flash_prefill_workspace_bytes(P_T, 0, P_T), dtype=torch.uint8, device=device)

    def floop():
        for b, d in enumerate(singles):
            qsa.qsa_flash_prefill(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], P_T, P_T, 0, None, outs1[b], ws1)
    med1, _ = gt(floop)
    fl = P_SEQ * flops_prefill(P_T, 0)
    # short prompts move more bytes than they compute: q in, out back (fp16), every cell's int8
    # K/V codes and fp16 scales once
    by = 2 * n_tok * HEADS * D * 2 + n_tok * 2 * 2 * (D + 8)
    res["prefill_batched"] = {"sequences": P_SEQ, "tokens_per_sequence": P_T, "pos0": 0, "us_per_call": med,
                              "us_per_call_min": mn, "tokens_per_s": n_tok / (med * 1e-6),
                              "us_for_single_calls": med1, "gflop": fl / 1e9, "bytes": by,
                              "hbm": _roof(by / (med * 1e-6) / 1e9, hbm_gbs, "GB/s", "hbm"),
                              "tensor": _roof(fl / (med * 1e-6) / 1e12, tf_burst, "TFLOP/s", "tensor"),
                              "call": "qsa_flash_prefill_batched (work list + mirror + dense: 3 launches), against "
                                      "64 qsa_flash_prefill calls in one graph"}
    del pool, singles, outs1
    res["hbm_calls"] = hbm_calls
    return res


def run_e2e(args, torch, qsa, device, stream, A, B, C, outA, outB, idsB, idsC, partC, nchC, xpC, wsB, wsC, pwsA,
            pwsB, nA, nB, nC, cap, dist):
    """The value's workload (12 identity-prefill layers, T=1984) through the public API with every
    layer's inputs copied from pinned host memory and its output copied back inside the timed region
    (copies overlap the kernels of other layers), then the same for the whole step (all three
    workloads) for context."""
    head = _e2e_leg(args, torch, qsa, device, stream, A, B, C, outA, outB, idsB, idsC, partC, nchC, xpC, wsB, wsC,
                    pwsA, pwsB, nA, nB, nC, cap, dist, "A")
    full = _e2e_leg(args, torch, qsa, device, stream, A, B, C, outA, outB, idsB, idsC, partC, nchC, xpC, wsB, wsC,
                    pwsA, pwsB, nA, nB, nC, cap, dist, "ABC")
    world = dist.get_world_size() if dist else 1
    return {"value": whole_job_rate(head["ms"], world), "unit": UNIT, "ms_per_12_layers": head["ms"],
            "h2d_bytes_per_step": head["h2d"], "d2h_bytes_per_step": head["d2h"],
            "whole_step": {"ms_per_step": full["ms"], "h2d_bytes_per_step": full["h2d"],
                           "d2h_bytes_per_step": full["d2h"],
                           "workload": "12 layers each of prefill T=1984 pos0=0, prefill T=1984 pos0=30000 and "
                                       "decode N=1 P=8192 (single launch), with host copies"}}


def _e2e_leg(args, torch, qsa, device, stream, A, B, C, outA, outB, idsB, idsC, partC, nchC, xpC, wsB, wsC, pwsA,
             pwsB, nA, nB, nC, cap, dist, which):
    """One end-to-end leg over the workloads named in `which`; returns ms per step and copy bytes."""
    hostA = [{k: v.cpu().pin_memory() for k, v in d.items()} for d in A]
    hostB = [{k: v.cpu().pin_memory() for k, v in d.items()} for d in B] if "B" in which else []
    hostC = [{k: v.cpu().pin_memory() for k, v in d.items()} for d in C] if "C" in which else []
    hOutA = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outA]
    hOutB = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outB] if "B" in which else []
    hXp = [torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in xpC] if "C" in which else []
    h2d = sum(v.numel() * v.element_size() for hs in (hostA, hostB, hostC) for d in hs for v in d.values())
    d2h = sum(o.numel() * o.element_size() for o in hOutA + hOutB + hXp)

    # one job per layer and workload: (device inputs, host inputs, compute, device output, host output)
    jobs = []
    for l in range(LAYERS):
        jobs.append((A[l], hostA[l], lambda d, l=l: qsa.qsa_flash_prefill(
            d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], nA, T_PREFILL, 0, None, outA[l], pwsA), outA[l], hOutA[l]))
    for l in range(LAYERS if "B" in which else 0):
        def run_b(d, l=l):
            qsa.qsa_select(d["q"], d["kq"], d["ksc"], nB, T_PREFILL, POS0_B, idsB[l], wsB)
            qsa.qsa_flash_prefill(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], nB, T_PREFILL, POS0_B, idsB[l],
                                  outB[l], pwsB)
        jobs.append((B[l], hostB[l], run_b, outB[l], hOutB[l]))
    for l in range(LAYERS if "C" in which else 0):
        def run_c(d, l=l):
            qsa.qsa_decode_layer(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], nC, N_DEC, P_DEC, idsC[l], xpC[l])
        jobs.append((C[l], hostC[l], run_c, xpC[l], hXp[l]))

    # Copies run on their own streams so that they overlap the kernels of other layers: job j's
    # inputs go up on h2d_s, its kernels run on the compute stream once they have landed, and its
    # output comes back on d2h_s.  A job's device buffers are reused next step only after its
    # kernels (for the inputs) and its read-back (for the output) are done.
    h2d_s, d2h_s = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    ev_in, ev_done, ev_out = [ev() for _ in jobs], [ev() for _ in jobs], [ev() for _ in jobs]
    for e in ev_done + ev_out:
        e.record(stream)

    def step():
        for j, (d, h, _, _, _) in enumerate(jobs):
            h2d_s.wait_event(ev_done[j])
            with torch.cuda.stream(h2d_s):
                for k in d:
                    d[k].copy_(h[k], non_blocking=True)
            ev_in[j].record(h2d_s)
        for j, (d, _, run, out, hout) in enumerate(jobs):
            stream.wait_event(ev_in[j])
            stream.wait_event(ev_out[j])
            run(d)
            ev_done[j].record(stream)
            d2h_s.wait_event(ev_done[j])
            with torch.cuda.stream(d2h_s):
                hout.copy_(out, non_blocking=True)
            ev_out[j].record(d2h_s)
        stream.wait_event(ev_out[-1])  # the step ends when its last result is back on the host

    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize(device)
    if dist:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    h2d_s.wait_event(e0)
    d2h_s.wait_event(e0)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1) / args.steps
    ms = max_over_ranks(ms, dist, device)
    return {"ms": ms, "h2d": h2d, "d2h": d2h}


def oracle_sample(seconds_budget=20.0):
    """Time the CPU oracle, as it stands, on a bounded sample of the same workload.

    The sample is taken from layer 0 of each workload:
      A: tokens of the identity prefill T=1984 pos0=0 at a fixed stride;
      B: the first tokens of the selected prefill T=1984 pos0=30000 (selection over
         ~31,984 cells, then attention);
      C: repeats of the decode token at P=8192.
    Each part first runs a small calibration sample, then a sample sized to fill about a
    third of `seconds_budget`.  The per-layer time of the full workload is extrapolated
    from the per-cell (A) and per-token (B, C) times of the sized samples.
    Returns (identity-prefill tokens/s per layer, description, cores, seconds spent)."""
    import oracle
    from int8_kv_top_gb300 import synth

    oracle.build()
    cores = os.cpu_count() or 1
    part = seconds_budget / 3.0
    spent = 0.0

    inpA = synth.layer_inputs(T_PREFILL, T_PREFILL, seed=5)

    def run_a(stride):
        toks = np.arange(0, T_PREFILL, stride, dtype=np.int32)
        t0 = time.perf_counter()
        oracle.prefill(inpA, T_PREFILL, 0, toks=toks)
        return time.perf_counter() - t0, int(sum(int(t) + 1 for t in toks)), len(toks)

    dt, cells, _ = run_a(124)
    spent += dt
    cells_all = sum(t + 1 for t in range(T_PREFILL))
    est_full = dt / cells * cells_all
    stride = max(1, int(np.ceil(est_full / part)))
    tA, cellsA, nA = run_a(stride)
    spent += tA
    full_A = tA / cellsA * cells_all

    def run_b(n_tok):
        inp = synth.layer_inputs(n_tok, POS0_B + n_tok, seed=105)
        t0 = time.perf_counter()
        oracle.prefill(inp, n_tok, POS0_B)
        return time.perf_counter() - t0

    nB0 = max(1, min(16, cores))
    dt = run_b(nB0)
    spent += dt
    nB = int(max(nB0, min(T_PREFILL, part / (dt / nB0))))
    tB = run_b(nB)
    spent += tB
    full_B = tB / nB * T_PREFILL

    inpC = synth.layer_inputs(N_DEC, P_DEC + N_DEC, seed=205)
    t0 = time.perf_counter()
    oracle.decode(inpC, N_DEC, P_DEC)
    dt = time.perf_counter() - t0
    spent += dt
    reps = int(max(1, min(200, part / max(dt, 1e-6))))
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.decode(inpC, N_DEC, P_DEC)
    tC = (time.perf_counter() - t0) / reps
    spent += tC * reps

    # the metric is the identity prefill's rate: T / (time of one identity-prefill layer)
    value = T_PREFILL / full_A
    desc = (f"identity prefill: layer 0, {nA} tokens (stride {stride}) of T=1984 pos0=0 in {tA:.2f}s, "
            f"extrapolated by causal cells to {full_A:.1f} s per layer (the value); for context, the selected "
            f"prefill at pos0=30000: the first {nB} tokens in {tB:.2f}s, {full_B:.1f} s per layer by tokens; decode "
            f"at P=8192: {tC * 1e3:.1f} ms per token ({reps} repeats); {cores} OpenMP threads")
    return value, desc, cores, spent


PROFILE_CASES = ("dense", "gather", "select", "decode", "decode_layer", "prep", "batched")


def run_profile_case(args):
    """Run one workload's API calls (args.steps times after args.warmup) for an ncu capture; prints
    nothing but a done line.  dense: prefill T=1984 pos0=0; select / gather: the select or the
    gathered prefill of T=1984 at pos0=30000; decode: select + partial + merge at N=1, P=8192.
    One layer's buffers, so the capture holds well under a GB on the device."""
    import torch

    from int8_kv_top_gb300 import qsa, synth
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    qsa.load()
    case = args.profile
    if case == "prep":
        pi = {k: torch.from_numpy(v).to(device) for k, v in synth.prep_inputs(T_PREFILL, seed=5).items()}
        n = T_PREFILL
        kq = torch.empty((n, 2, D), dtype=torch.int8, device=device)
        vq = torch.empty((n, 2, D), dtype=torch.int8, device=device)
        ksc = torch.empty((n, 2, 4), dtype=torch.float16, device=device)
        vsc = torch.empty((n, 2, 4), dtype=torch.float16, device=device)
        qcur = torch.empty((T_PREFILL, HEADS, D), dtype=torch.float16, device=device)
        for _ in range(args.warmup + args.steps):
            qsa.qsa_prep(pi["q_raw"], pi["k_raw"], pi["v_raw"], pi["q_gamma"], pi["k_gamma"], T_PREFILL, 0, n, qcur,
                         None, kq, ksc, vq, vsc)
        torch.cuda.synchronize(device)
        qsa.qsa_check_device_status()
        print(f"profile case prep: {args.warmup + args.steps} runs done", flush=True)
        return
    if case == "batched":  # 64 prompts of 128 tokens in one qsa_flash_prefill_batched call
        n_seq, tp = 64, 128
        parts = [synth.layer_inputs(tp, tp, seed=3500 + b) for b in range(n_seq)]
        pool = {k: torch.from_numpy(np.concatenate([pc[k] for pc in parts], axis=0)).to(device)
                for k in ("q", "kq", "vq", "ksc", "vsc")}
        seqs = torch.tensor([[b * tp, tp, 0, b * tp] for b in range(n_seq)], dtype=torch.int32, device=device)
        n_tok = n_seq * tp
        out = torch.empty((n_tok, HEADS, D), dtype=torch.float16, device=device)
        ws = torch.empty(qsa.qsa_flash_prefill_batched_workspace_bytes(n_seq, n_tok, tp), dtype=torch.uint8,
                         device=device)
        for _ in range(args.warmup + args.steps):
            qsa.qsa_flash_prefill_batched(pool["q"], pool["kq"], pool["vq"], pool["ksc"], pool["vsc"], n_tok, seqs,
                                          n_seq, n_tok, tp, None, out, ws)
        torch.cuda.synchronize(device)
        qsa.qsa_check_device_status()
        print(f"profile case batched: {args.warmup + args.steps} runs done", flush=True)
        return
    if case == "dense":
        T, pos0 = T_PREFILL, 0
    elif case in ("select", "gather"):
        T, pos0 = T_PREFILL, POS0_B
    else:
        T, pos0 = N_DEC, P_DEC
    n = pos0 + T
    d = {k: torch.from_numpy(v).to(device) for k, v in synth.layer_inputs(T, n, seed=5).items()}
    ids = torch.empty((T, 2, 2048), dtype=torch.int32, device=device)
    out = torch.empty((T, HEADS, D), dtype=torch.float16, device=device)
    sws = torch.empty(max(16, qsa.qsa_select_workspace_bytes(T, pos0, n)), dtype=torch.uint8, device=device)
    pws = torch.empty(qsa.qsa_flash_prefill_workspace_bytes(T, pos0, n), dtype=torch.uint8, device=device)
    cap = qsa.chunk_cap_for()
    part = torch.empty((T, cap, HEADS, 258), device=device)
    nch = torch.empty(T, dtype=torch.int32, device=device)
    xp = torch.empty((T, HEADS, D), device=device)
    if case == "gather":
        qsa.qsa_select(d["q"], d["kq"], d["ksc"], n, T, pos0, ids, sws)

    def once():
        if case == "decode_layer":
            qsa.qsa_decode_layer(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], n, T, pos0, ids, xp)
            return
        if case in ("select", "decode"):
            qsa.qsa_select(d["q"], d["kq"], d["ksc"], n, T, pos0, ids, sws)
        if case in ("dense", "gather"):
            qsa.qsa_flash_prefill(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], n, T, pos0,
                                  None if case == "dense" else ids, out, pws)
        if case == "decode":
            qsa.qsa_decode_partial(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], n, T, pos0, ids, part, nch, cap)
            qsa.qsa_merge(part, nch, T, cap, xp)
    for _ in range(args.warmup + args.steps):
        once()
    torch.cuda.synchronize(device)
    qsa.qsa_check_device_status()
    print(f"profile case {case}: {args.warmup + args.steps} runs done", flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-configuration timings")
    ap.add_argument("--profile", default=None, choices=PROFILE_CASES,
                    help="only run one workload's calls (--warmup + --steps times) for a profiler capture")
    ap.add_argument("--eager", action="store_true", help="time eager API calls instead of CUDA graph replays")
    ap.add_argument("--clocks-csv", default=None,
                    help="also keep the nvidia-smi samples of the timed region in this CSV ({rank} is replaced)")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.profile:
        run_profile_case(args)
        return

    if args.impl == "reference":
        # the reference arm is the CPU oracle, timed on the host cores; rank 0 only
        if rank != 0:
            return
        vals = []
        desc, cores = "", 1
        budget = max(3.0, min(20.0, 180.0 / max(1, args.warmup + args.steps)))
        for i in range(args.warmup + args.steps):
            v, desc, cores, _ = oracle_sample(budget)
            if i >= args.warmup:
                vals.append(v)
        v = statistics.median(vals)
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": 0, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": "same as the GPU arm, bounded sample per step"},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    line = run_ours(args, rank, world, local_rank)
    if rank == 0 and not args.no_cpu_baseline:
        v, desc, cores, secs = oracle_sample()
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc,
                                "seconds": secs}
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
