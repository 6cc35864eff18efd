"""Benchmark of the QSA layer hot path on GB300.

One step = 12 QSA layers (distinct, seeded synthetic buffers per layer) of each of:
  A  prefill  T=1984 at pos0=0      (identity: every causal cell)       qsa_flash_prefill
  B  prefill  T=1984 at pos0=30000  (31,984-cell cache, top-2048)       qsa_select + qsa_flash_prefill
  C  decode   N=1 at P=8192         (top-2048, 64-cell split)           qsa_select + qsa_decode_partial + qsa_merge
value = prefill tokens per second per layer over the whole step: (1984 + 1984) * 12 / (12 * step time).
The timed steps replay one CUDA graph per workload (captured from the same API calls); --eager
times the calls themselves.

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
UNIT = "tokens/s per layer"


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


def whole_job_rate(ms_per_step, world):
    """Prefill tokens/s per layer of the whole job: each of `world` replicas runs the full step
    (2 x 1984 prefill tokens in each of the 12 layers) in ms_per_step (the max over ranks)."""
    return 2 * T_PREFILL * LAYERS / (ms_per_step * 1e-3) / LAYERS * world


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
    launches_per_step = LAYERS * (2 + 6 + 4)

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
            qsa.qsa_select(d["q"], d["kq"], d["ksc"], nC, N_DEC, P_DEC, idsC[l], wsC)
            mark("Cp")
            qsa.qsa_decode_partial(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], nC, N_DEC, P_DEC, idsC[l], partC,
                                   nchC, cap)
            mark("Cm")
            qsa.qsa_merge(partC, nchC, N_DEC, cap, xpC[l])
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
    fam = {"dense_prefill": 0.0, "select_B": 0.0, "gather_prefill": 0.0, "select_C": 0.0, "decode_partial": 0.0,
           "merge": 0.0}
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
                fam["select_C"] += dt
            elif n == "Cp":
                fam["decode_partial"] += dt
            elif n == "Cm":
                fam["merge"] += dt
            del nxt
    fam = {k: v / max(1, len(all_marks)) for k, v in fam.items()}  # ms per step (12 launches each)
    # per-workload times of the timed steps: graph replays when available, else the eager marks
    if graphs:
        sec = {"A": sec_ms[0], "B": sec_ms[1], "C": sec_ms[2]}
    else:
        sec = {"A": fam["dense_prefill"], "B": fam["select_B"] + fam["gather_prefill"],
               "C": fam["select_C"] + fam["decode_partial"] + fam["merge"]}

    # ---- e2e: same step through the public API from pinned host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, torch, qsa, device, stream, A, B, C, outA, outB, idsB, idsC, partC, nchC, xpC, wsB, wsC,
                      pwsA, pwsB, nA, nB, nC, cap, dist)

    hbm_gbs, bf16_tf, bf16_tf_sus, peak_src = read_peaks()
    flopA = flops_prefill(T_PREFILL, 0)
    flopB = flops_prefill(T_PREFILL, POS0_B)
    per_launch = {
        "dense_prefill": {"bound": "tensor", "achieved": flopA / (sec["A"] / LAYERS * 1e-3) / 1e12,
                          "peak": bf16_tf_sus, "unit": "TFLOP/s"},
        "gather_prefill": {"bound": "tensor", "achieved": flopB / (fam["gather_prefill"] / LAYERS * 1e-3) / 1e12,
                           "peak": bf16_tf_sus, "unit": "TFLOP/s",
                           # the selected rows are gathered from L2: T x 2 groups x 2048 cells x 1 KB (K^ + V^ fp16)
                           "l2_gather_gbs": T_PREFILL * 2 * 2048 * 1024 / (fam["gather_prefill"] / LAYERS * 1e-3) / 1e9},
    }
    for v in per_launch.values():
        v["frac"] = v["achieved"] / v["peak"]
    for k, v in per_launch.items():
        v["traffic"] = recorded_traffic(KERNEL_OF_FAMILY[k])
    dominant = max(("dense_prefill", "gather_prefill", "select_B"), key=lambda k: fam[k])
    if dominant == "select_B":
        # select moves the score matrix through HBM: written once (fp16) and read once, plus K codes
        T_sel = T_PREFILL
        n_avg = POS0_B + (T_PREFILL + 1) / 2
        bytes_sel = 2 * T_sel * n_avg * 2 * 2 + 2 * nB * (256 + 8) + 2 * nB * 512
        roof = {"bound": "hbm", "achieved": bytes_sel / (fam["select_B"] / LAYERS * 1e-3) / 1e9, "peak": hbm_gbs,
                "unit": "GB/s", "kernel": "qsa_select (4 launches)"}
        roof["frac"] = roof["achieved"] / roof["peak"]
    else:
        roof = dict(per_launch[dominant])
        roof["kernel"] = dominant
    roof["traffic"] = recorded_traffic(KERNEL_OF_FAMILY.get(dominant, ""))
    roof["traffic_unit"] = "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)"
    roof["peak_source"] = f"{peak_src}, sustained bf16 (f16 same rate)" if roof["unit"] == "TFLOP/s" else peak_src

    value = whole_job_rate(ms_step, world)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16 operands, f32 accumulate", "data": "synthetic (seeded; q~N(0,1) fp16, int8 K/V uniform "
        "[-127,127], fp16 scales U[0.005,0.02])",
        "config": {"workload": "12 QSA layers x {prefill T=1984 pos0=0 (identity); prefill T=1984 pos0=30000 "
                               "(31984-cell cache, top-2048); decode N=1 P=8192}", "layers": LAYERS,
                   "heads": "2 KV x 12 q, dim 256", "l2": "inputs larger than L2 (12 distinct layer buffer sets)",
                   "parallelism": f"replicas x{world}"},
        "breakdown_ms_per_step": fam,
        "breakdown_timing": "eager calls, CUDA events between them",
        "timing": "CUDA graph replay per workload" if graphs else "eager calls",
        "workload_ms_per_step": sec,
        "prefill_identity_us_per_layer": sec["A"] / LAYERS * 1e3,
        "prefill_selected_us_per_layer": sec["B"] / LAYERS * 1e3,
        "decode_us_per_token_per_layer": sec["C"] / LAYERS * 1e3 / N_DEC,
        "roofline": roof, "roofline_per_kernel": per_launch,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks, "e2e": e2e,
    }
    return line


def run_e2e(args, torch, qsa, device, stream, A, B, C, outA, outB, idsB, idsC, partC, nchC, xpC, wsB, wsC, pwsA,
            pwsB, nA, nB, nC, cap, dist):
    """Same step with every layer's inputs copied from pinned host memory and outputs copied back,
    all inside the timed region; copies overlap the kernels of other layers."""
    hostA = [{k: v.cpu().pin_memory() for k, v in d.items()} for d in A]
    hostB = [{k: v.cpu().pin_memory() for k, v in d.items()} for d in B]
    hostC = [{k: v.cpu().pin_memory() for k, v in d.items()} for d in C]
    hOutA = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outA]
    hOutB = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outB]
    hXp = [torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in xpC]
    h2d = sum(v.numel() * v.element_size() for hs in (hostA, hostB, hostC) for d in hs for v in d.values())
    d2h = sum(o.numel() * o.element_size() for o in hOutA + hOutB + hXp)

    # one job per layer and workload: (device inputs, host inputs, compute, device output, host output)
    jobs = []
    for l in range(LAYERS):
        jobs.append((A[l], hostA[l], lambda d, l=l: qsa.qsa_flash_prefill(
            d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], nA, T_PREFILL, 0, None, outA[l], pwsA), outA[l], hOutA[l]))
    for l in range(LAYERS):
        def run_b(d, l=l):
            qsa.qsa_select(d["q"], d["kq"], d["ksc"], nB, T_PREFILL, POS0_B, idsB[l], wsB)
            qsa.qsa_flash_prefill(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], nB, T_PREFILL, POS0_B, idsB[l],
                                  outB[l], pwsB)
        jobs.append((B[l], hostB[l], run_b, outB[l], hOutB[l]))
    for l in range(LAYERS):
        def run_c(d, l=l):
            qsa.qsa_select(d["q"], d["kq"], d["ksc"], nC, N_DEC, P_DEC, idsC[l], wsC)
            qsa.qsa_decode_partial(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], nC, N_DEC, P_DEC, idsC[l], partC,
                                   nchC, cap)
            qsa.qsa_merge(partC, nchC, N_DEC, cap, xpC[l])
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
    world = dist.get_world_size() if dist else 1
    value = whole_job_rate(ms, world)
    return {"value": value, "unit": UNIT, "ms_per_step": ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


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
    Returns (tokens/s per layer, description, cores, seconds spent)."""
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

    per_layer = full_A + full_B + tC
    value = 2 * T_PREFILL / per_layer
    desc = (f"layer 0: {nA} tokens (stride {stride}) of T=1984 pos0=0 in {tA:.2f}s; the first {nB} tokens of "
            f"T=1984 pos0=30000 in {tB:.2f}s; {reps} x the decode token at P=8192 in {tC * reps:.2f}s; per-layer "
            f"time extrapolated by cells (A) and tokens (B, C); {cores} OpenMP threads")
    return value, desc, cores, spent


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true", help="time eager API calls instead of CUDA graph replays")
    ap.add_argument("--clocks-csv", default=None,
                    help="also keep the nvidia-smi samples of the timed region in this CSV ({rank} is replaced)")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

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
