"""Benchmark of the group-wise affine-quantized multi-row matmul on GB300.

Workload (MLP up-projection shape): K=5120, N=17408, 4-bit codes, group 32,
bf16 out, M in {1, 2, 4, 8, 16} rows. One step = 40 qmm_forward calls: every
M on each of 8 independent weight copies (8 x 55.7 MB = 446 MB > 3x the 129 MB
L2), in a fixed rotation so no call reads weights the previous call touched.
Inputs are seeded synthetic data (datagen), resident in HBM before timing.

Metric: effective HBM GB/s = (packed codes + fp16 scales + fp16 biases + bf16 x
+ bf16 y) bytes / time, plus us/call and GB/s per M.

The same line carries `per_config`: us/call, GB/s and the fraction of the
measured HBM peak for the other named configurations, each over rotating device
copies of its weights larger than L2 and timed by CUDA-graph replay: pr1_ref
(M=1, 2048 x 2048, 4-bit g64, fp32 out; also with direct stream launches),
down_longk (17408 -> 5120, 4-bit g64, splits 1/2/4/8/automatic x M 1/8/16),
mixed_widths (5120 -> 6144, 5/6/8-bit g32, M=8), the 4/5/6/8-bit widths on the
mlp_up shape (M=8) and banked (36 banks of
2048 -> 8192, 4-bit g64, M 1 and 16, per bank set).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl qmm|reference]

--impl reference times the CPU oracle (float64 C++) on the same workload (a
bounded sample per step). Under torchrun each rank runs an independent replica
(the op has no exchange step); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import subprocess
import tempfile
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import datagen  # noqa: E402

WORKLOAD = "mlp_up"
MS = [1, 2, 4, 8, 16]
COPIES = 8
METRIC = "qmm effective HBM GB/s (codes+scales+biases+x+y bytes / time), M=1,2,4,8,16"

# DRAM bytes per main-kernel launch measured with ncu (dram__bytes_read.sum +
# dram__bytes_write.sum) on this workload, keyed by M, and the hash of the
# kernel sources' code (comments ignored) they were measured on. If the code
# changes, traffic is reported as null until re-measured.
TRAFFIC = {"source_sha": "2524775ed830a768",
           "per_M": {"1": 55773696, "2": 55780096, "4": 55800064, "8": 55841024, "16": 55920896}}


def _code_only(text: str) -> str:
    """C++/CUDA source with comments and blank space removed (string literals
    in these sources hold no comment markers), so that edits to comments alone
    keep the hash."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_sha() -> str:
    """Hash of the kernel sources' code (comments ignored), tying the ncu DRAM
    traffic figures below to the kernels they were measured on."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_affine_quantized_group_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                h.update(name.encode() + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def algorithmic_bytes(M: int, K: int, N: int, bits: int, group: int, out_bytes: int) -> int:
    codes = N * K * bits // 8
    sb = N * (K // group) * 2 * 2
    return codes + sb + M * K * 2 + M * N * out_bytes


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


# ---------------------------------------------------------------------------
# distributed (replicas only: barrier + max of the timed region)
# ---------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_init(ws: int, backend: str):
    if ws <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend=backend)
    return dist


def aggregate(dist, value_local_units: float, seconds_local: float):
    """Whole-job throughput: units summed over ranks / max time over ranks."""
    if dist is None:
        return value_local_units, seconds_local
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([seconds_local], dtype=torch.float64, device=dev)
    u = torch.tensor([value_local_units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(u.item()), float(t.item())


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
        # raw samples; the summary goes into the JSON line
        self.path = os.path.join(tempfile.gettempdir(), f"qmm_bench_clocks_rank{gpu_index}_{os.getpid()}.csv")

    def start(self):
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        # "under load": samples within 30% of the highest observed clock (idle gaps excluded)
        top = max(sm) if sm else 0.0
        load = [v for v in sm if v >= 0.7 * top] or sm
        return {"sm_mhz": float(np.median(load)) if load else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# Every named configuration, timed the same way (a JSON object in the line)
# ---------------------------------------------------------------------------
L2_BYTES = 129 * 2 ** 20


def _time_step(step, reps, stream, graph=True, passes=3):
    """Seconds per step(): warm-up, then (optionally) one CUDA-graph capture of
    step() replayed `reps` times; the fastest of `passes` timed passes."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
    torch.cuda.synchronize()
    g = None
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step()
        torch.cuda.synchronize()
    best = float("inf")
    for _ in range(passes):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            (g.replay() if g is not None else step())
            e0.record(stream)
            for _ in range(reps):
                (g.replay() if g is not None else step())
            e1.record(stream)
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1) / 1e3 / reps)
    del g
    return best


def _dev_copies(name, bits, M, banks=1, min_bytes=3 * L2_BYTES):
    """x on the device and enough device copies of the workload's weights
    (clones of one seeded copy per bank) that one rotation exceeds `min_bytes`."""
    import torch
    wl = datagen.WORKLOADS[name]
    K, N, group = wl["K"], wl["N"], wl["group"]
    inp = datagen.gen_qmm(datagen.workload_seed(name) + bits, M, K, N, bits, group, banks=banks)
    dev = torch.device("cuda", torch.cuda.current_device())
    x = torch.from_numpy(inp.x.view(np.int16)).to(dev).view(torch.bfloat16)
    base = [(torch.from_numpy(inp.words[i].view(np.int32)).to(dev),
             torch.from_numpy(inp.scales[i].view(np.int16)).to(dev).view(torch.float16),
             torch.from_numpy(inp.biases[i].view(np.int16)).to(dev).view(torch.float16)) for i in range(banks)]
    per_set = banks * algorithmic_bytes(0, K, N, bits, group, 0)
    sets = max(1, -(-min_bytes // per_set))
    copies = [base] + [[tuple(t.clone() for t in bk) for bk in base] for _ in range(sets - 1)]
    return x, copies, (K, N, group)


def run_per_config(q, peaks, stream):
    """us/call (or per bank set), effective GB/s and fraction of the measured HBM
    peak for every named configuration other than the headline's."""
    import torch
    peak = peaks["hbm_gbs"]
    res = {}

    def entry(sec, nbytes, extra=None):
        d = {"us": round(sec * 1e6, 3), "gbs": round(nbytes / sec / 1e9, 1), "frac": round(nbytes / sec / 1e9 / peak, 4)}
        if extra:
            d.update(extra)
        return d

    # pr1_ref: M=1, 2048 x 2048, 4-bit g64, fp32 out; direct stream launches and graph replay
    x, copies, (K, N, group) = _dev_copies("pr1_ref", 4, 1)
    plan = q.Plan(K, N, 4, group, max_M=1, out_dtype="f32", splits=0)
    out = torch.empty((1, N), dtype=torch.float32, device=x.device)

    def step_pr1():
        for c in copies:
            q.forward(plan, x, c[0][0], c[0][1], c[0][2], out, stream=stream)
    nb = algorithmic_bytes(1, K, N, 4, group, 4)
    reps = max(5, 2000 // len(copies))
    sg = _time_step(step_pr1, reps, stream, graph=True) / len(copies)
    sd = _time_step(step_pr1, reps, stream, graph=False) / len(copies)
    res["pr1_ref"] = {"workload": f"M=1 K={K} N={N} 4-bit g{group} f32 out", "splits": plan.info()["splits"],
                      "copies": len(copies), "graph": entry(sg, nb), "stream": entry(sd, nb)}
    assert plan.error_flags() == 0
    del copies, plan

    # down_longk: 17408 -> 5120, 4-bit g64, bf16 out, splits 1/2/4/8/auto x M 1/8/16
    x, copies, (K, N, group) = _dev_copies("down_longk", 4, 16)
    dl = {"workload": f"K={K} N={N} 4-bit g{group} bf16 out", "copies": len(copies)}
    for splits in (1, 2, 4, 8, 0):
        plan = q.Plan(K, N, 4, group, max_M=16, out_dtype="bf16", splits=splits)
        row = {"splits_used": plan.info()["splits"]}
        for M in (1, 8, 16):
            out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)

            def step_dl():
                for c in copies:
                    q.forward(plan, x[:M], c[0][0], c[0][1], c[0][2], out, stream=stream)
            sec = _time_step(step_dl, max(5, 400 // len(copies)), stream) / len(copies)
            row[str(M)] = entry(sec, algorithmic_bytes(M, K, N, 4, group, 2))
        assert plan.error_flags() == 0
        dl["auto" if splits == 0 else f"splits={splits}"] = row
        del plan
    res["down_longk"] = dl
    del copies

    # mixed widths: 5120 -> 6144, 5/6/8-bit g32, M=8, bf16 out, automatic splits
    mw = {}
    for bits in (5, 6, 8):
        x, copies, (K, N, group) = _dev_copies("mixed_widths", bits, 8)
        plan = q.Plan(K, N, bits, group, max_M=8, out_dtype="bf16", splits=0)
        out = torch.empty((8, N), dtype=torch.bfloat16, device=x.device)

        def step_mw():
            for c in copies:
                q.forward(plan, x, c[0][0], c[0][1], c[0][2], out, stream=stream)
        sec = _time_step(step_mw, max(5, 400 // len(copies)), stream) / len(copies)
        mw[f"{bits}-bit"] = entry(sec, algorithmic_bytes(8, K, N, bits, group, 2),
                                  {"splits": plan.info()["splits"], "copies": len(copies)})
        assert plan.error_flags() == 0
        del copies, plan
    res["mixed_widths"] = {"workload": "M=8 K=5120 N=6144 g32 bf16 out", **mw}

    # the same code widths on the headline's shape (5120 -> 17408, g32, M=8), so
    # that the odd widths compare with 4-bit codes at equal problem size
    ws_ = {}
    for bits in (4, 5, 6, 8):
        x, copies, (K, N, group) = _dev_copies("mlp_up", bits, 8)
        plan = q.Plan(K, N, bits, group, max_M=8, out_dtype="bf16", splits=0)
        out = torch.empty((8, N), dtype=torch.bfloat16, device=x.device)

        def step_ws():
            for c in copies:
                q.forward(plan, x, c[0][0], c[0][1], c[0][2], out, stream=stream)
        sec = _time_step(step_ws, max(5, 400 // len(copies)), stream) / len(copies)
        ws_[f"{bits}-bit"] = entry(sec, algorithmic_bytes(8, K, N, bits, group, 2),
                                   {"splits": plan.info()["splits"], "copies": len(copies)})
        assert plan.error_flags() == 0
        del copies, plan
    res["widths_at_mlp_up_shape"] = {"workload": "M=8 K=5120 N=17408 g32 bf16 out", **ws_}

    # banked: 36 x (2048 -> 8192), 4-bit g64, shared x, M 1 and 16, per bank set
    x, sets, (K, N, group) = _dev_copies("banked", 4, 16, banks=36, min_bytes=2 * L2_BYTES)
    B = 36
    plan = q.Plan(K, N, 4, group, max_M=16, out_dtype="bf16", splits=0, max_banks=B)
    bk = {"workload": f"{B} banks x (K={K} N={N} 4-bit g{group}) shared x, bf16 out", "bank_sets": len(sets),
          "splits": plan.info()["splits"]}
    for M in (1, 16):
        outs = [torch.empty((M, N), dtype=torch.bfloat16, device=x.device) for _ in range(B)]

        def step_bk():
            for st in sets:
                q.forward_banked(plan, x[:M], [c[0] for c in st], [c[1] for c in st], [c[2] for c in st], outs,
                                 stream=stream)
        sec = _time_step(step_bk, max(5, 100 // len(sets)), stream) / len(sets)
        bk[str(M)] = entry(sec, B * algorithmic_bytes(M, K, N, 4, group, 2), {"unit": "per bank set"})
    assert plan.error_flags() == 0
    res["banked"] = bk
    del sets, plan
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def run_gpu(args, ws, rank, local):
    import torch
    from bit_affine_quantized_group_gb300 import _build
    _build.build()
    import bit_affine_quantized_group_gb300 as q

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = dist_init(ws, "nccl")
    wl = datagen.WORKLOADS[WORKLOAD]
    K, N, bits, group = wl["K"], wl["N"], 4, wl["group"]

    inp = datagen.gen_qmm(datagen.workload_seed(WORKLOAD), 16, K, N, bits, group, banks=COPIES)
    x_host = inp.x
    x = torch.from_numpy(x_host.view(np.int16)).to(dev).view(torch.bfloat16)
    W = [torch.from_numpy(inp.words[i].view(np.int32)).to(dev) for i in range(COPIES)]
    S = [torch.from_numpy(inp.scales[i].view(np.int16)).to(dev).view(torch.float16) for i in range(COPIES)]
    B = [torch.from_numpy(inp.biases[i].view(np.int16)).to(dev).view(torch.float16) for i in range(COPIES)]
    del inp
    plan = q.Plan(K, N, bits, group, max_M=16, out_dtype="bf16", splits=0, device=dev)
    info = plan.info()
    outs = {M: torch.empty((M, N), dtype=torch.bfloat16, device=dev) for M in MS}
    kernels_per_call = 1 + (1 if info["splits"] > 1 else 0)   # the main kernel (+ the split-K reduce)

    # one step: call j uses M = MS[j % 5] and weight copy j % 8 (all 40 pairs)
    calls = [(MS[j % len(MS)], j % COPIES) for j in range(len(MS) * COPIES)]
    step_bytes = sum(algorithmic_bytes(M, K, N, bits, group, 2) for M, _ in calls)
    stream = torch.cuda.Stream(device=dev)

    def step(call_list):
        for M, c in call_list:
            q.forward(plan, x[:M], W[c], S[c], B[c], outs[M], stream=stream)

    def timed(call_list, steps, warmup, use_graph):
        with torch.cuda.stream(stream):
            for _ in range(max(warmup, 3)):
                step(call_list)
        torch.cuda.synchronize()
        graph = None
        if use_graph:
            try:
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, stream=stream):
                    step(call_list)
                torch.cuda.synchronize()
                with torch.cuda.stream(stream):
                    for _ in range(3):
                        graph.replay()
                torch.cuda.synchronize()
            except Exception as e:   # capture unsupported: time direct launches
                sys.stderr.write(f"graph capture failed ({e}); timing direct launches\n")
                graph = None
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(steps):
                if graph is not None:
                    graph.replay()
                else:
                    step(call_list)
            e1.record(stream)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        return e0.elapsed_time(e1) / 1e3, graph is not None

    peaks = load_peaks()
    use_graph = not args.no_graph

    # per-M loops (8 calls, one per weight copy)
    per_m = {}
    for M in MS:
        cl = [(M, c) for c in range(COPIES)]
        reps = max(20, args.steps // 4)
        sec, _ = timed(cl, reps, args.warmup, use_graph)
        us = sec / (reps * COPIES) * 1e6
        gbs = algorithmic_bytes(M, K, N, bits, group, 2) / (us * 1e-6) / 1e9
        per_m[str(M)] = {"us_per_call": round(us, 3), "gbs": round(gbs, 1),
                         "frac": round(gbs / peaks["hbm_gbs"], 4)}

    # headline: K steps of the full 40-call sweep, clocks sampled meanwhile
    clocks = ClockSampler(local)
    clocks.start()
    sec, graphed = timed(calls, args.steps, args.warmup, use_graph)
    clk = clocks.stop()
    units_local = step_bytes * args.steps / 1e9
    units, sec_max = aggregate(dist, units_local, sec)
    value = units / sec_max
    ms_per_step = sec_max / args.steps * 1e3

    # end to end through the public call with host buffers: each step copies its
    # input x (pinned host -> device, once per step: every call of the step reads
    # rows of the same x), runs the 40 calls, and reads every call's output back
    # into pinned host memory. The 40 outputs of a step are consecutive views of
    # one device buffer, read back with one copy on a second stream once the step's
    # last call is done, so the read-back overlaps the next step's calls (two
    # output buffers alternate between steps; nothing is inserted between two
    # calls of a step, which would break their programmatic-dependent launch
    # overlap). The timed region ends when the last step's read-back has landed.
    x_pin = torch.from_numpy(x_host.view(np.int16)).pin_memory()
    x_dev = torch.empty((16, K), dtype=torch.int16, device=dev)
    total_rows = sum(M for M, _ in calls)
    y_dev = [torch.empty((total_rows * N,), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    y_host = [torch.empty((total_rows * N,), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    outs_e2e = []
    for buf in y_dev:
        views, off = [], 0
        for M, _ in calls:
            views.append(buf[off:off + M * N].view(M, N))
            off += M * N
        outs_e2e.append(views)
    d2h_stream = torch.cuda.Stream(device=dev)
    calls_done = [torch.cuda.Event() for _ in range(2)]
    read_done = [torch.cuda.Event() for _ in range(2)]
    e2e_steps = max(5, min(args.steps, 200))
    h2d = 16 * K * 2
    d2h = sum(M * N * 2 for M, _ in calls)

    def e2e_step(i):
        b = i % 2
        with torch.cuda.stream(stream):
            stream.wait_event(read_done[b])      # the buffer's previous read-back has landed
            x_dev.copy_(x_pin, non_blocking=True)
            for j, (M, c) in enumerate(calls):
                q.forward(plan, x_dev[:M].view(torch.bfloat16), W[c], S[c], B[c], outs_e2e[b][j], stream=stream)
            calls_done[b].record(stream)
        with torch.cuda.stream(d2h_stream):
            d2h_stream.wait_event(calls_done[b])
            y_host[b].copy_(y_dev[b], non_blocking=True)
            read_done[b].record(d2h_stream)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step(i)
    stream.synchronize()
    d2h_stream.synchronize()
    e2e_sec = time.perf_counter() - t0
    e2e_units, e2e_max = aggregate(dist, step_bytes * e2e_steps / 1e9, e2e_sec)
    e2e_value = e2e_units / e2e_max
    # the outputs read back are the call results (check against the device copy)
    last = (e2e_steps - 1) % 2
    if not torch.equal(y_host[last], y_dev[last].cpu()):
        raise RuntimeError("end-to-end read-back differs from the device result")

    flags = plan.error_flags()
    if flags != 0:
        raise RuntimeError(f"kernel reported a bounded-wait timeout (flags={flags})")

    per_config = None
    if not args.no_per_config:
        del W, S, B
        torch.cuda.empty_cache()
        per_config = run_per_config(q, peaks, stream)

    if rank != 0:
        return
    traffic = None
    if TRAFFIC["source_sha"] == kernel_source_sha() and TRAFFIC["per_M"]:
        traffic = float(np.mean([TRAFFIC["per_M"][str(M)] for M in MS]))
    cpu = cpu_baseline(K, N, bits, group) if ws == 1 else None
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded: uniform codes, fp16 scales U[0.002,0.02], biases -8*s+N(0,1e-3), x~N(0,1) bf16)",
        "config": {"workload": f"{WORKLOAD}: K={K} N={N} bits={bits} group={group} out=bf16 M=1,2,4,8,16",
                   "calls_per_step": len(calls), "weight_copies": COPIES,
                   "l2": f"inputs larger than L2: {COPIES} rotating weight copies "
                         f"({COPIES * algorithmic_bytes(0, K, N, bits, group, 0) / 1e6:.0f} MB > 3x 129 MB L2)",
                   "launch": "cuda_graph" if graphed else "direct", "splits": info["splits"],
                   "stages": info["stages"], "parallelism": f"replicas x{ws}", "accumulate": "fp32"},
        "per_M": per_m,
        "per_config": per_config,
        "roofline": {"bound": "hbm", "achieved": round(value / ws, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(value / ws / peaks["hbm_gbs"], 4), "traffic": traffic,
                     "peak_source": peaks["source"], "kernel": "qmm_main_kernel (one launch per call: weight stream, activation staging and contraction)"},
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps, "launch": "direct",
                "copies": "x host->device once per step; every call's y device->host in one copy per step, overlapping the next step's calls"},
        "gpu_launches": kernels_per_call * len(calls) * args.steps,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# CPU oracle (reported baseline and reference arm)
# ---------------------------------------------------------------------------
def oracle_sample(K, N, bits, group, ncols):
    """One bounded sample of the workload on the oracle: every M, `ncols`
    output columns. Returns (seconds, algorithmic bytes of that sample)."""
    import oracle
    oracle.build()
    inp = datagen.gen_qmm(datagen.workload_seed(WORKLOAD), 16, K, N, bits, group)
    cols = np.arange(ncols, dtype=np.int64)
    frac = ncols / N
    t0 = time.perf_counter()
    for M in MS:
        oracle.qmm_f64_cols(inp.x[:M], inp.words[0], inp.scales[0], inp.biases[0], K, N, bits, group, cols)
    sec = time.perf_counter() - t0
    nbytes = sum(int(algorithmic_bytes(M, K, N, bits, group, 2) * frac) for M in MS)
    return sec, nbytes


def cpu_baseline(K, N, bits, group):
    import oracle
    oracle.build()
    ncols = N
    total_sec, total_bytes, runs = 0.0, 0, 0
    while total_sec < 10.0 and runs < 50:
        sec, nb = oracle_sample(K, N, bits, group, ncols)
        total_sec += sec
        total_bytes += nb
        runs += 1
    return {"value": round(total_bytes / total_sec / 1e9, 4), "unit": "GB/s", "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": f"{runs} full sweeps of M=1,2,4,8,16 over all {N} columns ({total_sec:.1f} s)"}


def run_reference(args, ws, rank):
    if rank != 0:
        return
    import oracle
    oracle.build()
    wl = datagen.WORKLOADS[WORKLOAD]
    K, N, bits, group = wl["K"], wl["N"], 4, wl["group"]
    # bounded sample per step: all M values on the first `ncols` output columns,
    # sized so that warmup + steps take about 90 s of oracle time in total
    t_cal, _ = oracle_sample(K, N, bits, group, 256)
    per_step = min(3.0, 90.0 / max(1, args.steps + args.warmup))
    ncols = int(256 * per_step / max(t_cal, 1e-6)) // 16 * 16
    ncols = max(16, min(N, ncols))
    for _ in range(args.warmup):
        oracle_sample(K, N, bits, group, ncols)
    tot_sec, tot_bytes = 0.0, 0
    for _ in range(args.steps):
        sec, nb = oracle_sample(K, N, bits, group, ncols)
        tot_sec += sec
        tot_bytes += nb
    value = tot_bytes / tot_sec / 1e9
    sample = f"per step: M=1,2,4,8,16 on {ncols} of {N} output columns (bytes scaled to the sample)"
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(tot_sec / max(1, args.steps) * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (same seeded inputs as the GPU arm)",
        "config": {"workload": f"{WORKLOAD}: K={K} N={N} bits={bits} group={group} out=bf16 M=1,2,4,8,16",
                   "parallelism": "CPU oracle, OpenMP over columns"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.max_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ncu_case(args):
    """A small, untimed case for profilers: `calls` qmm_forward calls with M rows on
    one weight copy of the workload (about 60 MB on the device)."""
    import torch
    from bit_affine_quantized_group_gb300 import _build
    _build.build()
    import bit_affine_quantized_group_gb300 as q
    wl = datagen.WORKLOADS[args.case_workload]
    bits = args.case_bits or wl["bits"][0]
    K, N, group = wl["K"], wl["N"], wl["group"]
    M = args.ncu_case
    B = wl["banks"]
    inp = datagen.gen_qmm(datagen.workload_seed(args.case_workload), M, K, N, bits, group, banks=B)
    x = torch.from_numpy(inp.x.view(np.int16)).cuda().view(torch.bfloat16)
    W = [torch.from_numpy(inp.words[i].view(np.int32)).cuda() for i in range(B)]
    S = [torch.from_numpy(inp.scales[i].view(np.int16)).cuda().view(torch.float16) for i in range(B)]
    Bi = [torch.from_numpy(inp.biases[i].view(np.int16)).cuda().view(torch.float16) for i in range(B)]
    plan = q.Plan(K, N, bits, group, max_M=M, out_dtype=wl["out"], splits=args.case_splits, max_banks=B)
    outs = [torch.empty((M, N), dtype=plan.out_dtype, device="cuda") for _ in range(B)]
    for _ in range(args.calls):
        if B == 1:
            q.forward(plan, x, W[0], S[0], Bi[0], outs[0])
        else:
            q.forward_banked(plan, x, W, S, Bi, outs)
    torch.cuda.synchronize()
    print(f"ncu case ok: {args.case_workload} M={M} bits={bits} splits={plan.info()['splits']} calls={args.calls}")


COST_TABLE_CASES = [("mlp_up", 4), ("down_longk", 4), ("mixed_widths", 5), ("mixed_widths", 6),
                    ("mixed_widths", 8), ("lm_head", 8)]


def run_cost_table(args):
    """Per-M cost table (us/call for every M in 1..16) of the named workloads,
    for a row-width chooser: CUDA-graph replay over enough rotating weight
    copies to exceed 3x L2 (device clones of one generated copy), one JSON line."""
    import torch
    from bit_affine_quantized_group_gb300 import _build
    _build.build()
    import bit_affine_quantized_group_gb300 as q
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device=dev)
    table = {}
    for name, bits in COST_TABLE_CASES:
        wl = datagen.WORKLOADS[name]
        K, N, group = wl["K"], wl["N"], wl["group"]
        inp = datagen.gen_qmm(datagen.workload_seed(name) + bits, 16, K, N, bits, group)
        x = torch.from_numpy(inp.x.view(np.int16)).to(dev).view(torch.bfloat16)
        w0 = torch.from_numpy(inp.words[0].view(np.int32)).to(dev)
        s0 = torch.from_numpy(inp.scales[0].view(np.int16)).to(dev).view(torch.float16)
        b0 = torch.from_numpy(inp.biases[0].view(np.int16)).to(dev).view(torch.float16)
        del inp
        per_copy = algorithmic_bytes(16, K, N, bits, group, 2)
        copies = max(1, -(-3 * 129 * 2 ** 20 // per_copy))
        W = [w0] + [w0.clone() for _ in range(copies - 1)]
        S = [s0] + [s0.clone() for _ in range(copies - 1)]
        B = [b0] + [b0.clone() for _ in range(copies - 1)]
        plan = q.Plan(K, N, bits, group, max_M=16, out_dtype="bf16", splits=0, device=dev)
        row = {}
        for M in range(1, 17):
            out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)

            def step():
                for c in range(copies):
                    q.forward(plan, x[:M], W[c], S[c], B[c], out, stream=stream)
            with torch.cuda.stream(stream):
                for _ in range(3):
                    step()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step()
            # the fastest of three timed passes (a pass can catch a transient stall)
            reps = max(3, 400 // copies)
            us = float("inf")
            for _ in range(3):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(stream):
                    g.replay()
                    e0.record(stream)
                    for _ in range(reps):
                        g.replay()
                    e1.record(stream)
                torch.cuda.synchronize()
                us = min(us, e0.elapsed_time(e1) * 1e3 / (reps * copies))
            row[str(M)] = {"us_per_call": round(us, 3),
                           "gbs": round(algorithmic_bytes(M, K, N, bits, group, 2) / us / 1e3, 1)}
            del g, out
        assert plan.error_flags() == 0
        table[f"{name}:{bits}-bit"] = {"K": K, "N": N, "group": group, "splits": plan.info()["splits"],
                                       "copies": copies, "per_M": row}
        del W, S, B, w0, s0, b0, plan
        torch.cuda.empty_cache()
    # fused gate/up (SwiGLU) on the mlp_up shape: one fused call against the two
    # separate projections it replaces
    wl = datagen.WORKLOADS["mlp_up"]
    K, N, group, bits = wl["K"], wl["N"], wl["group"], 4
    gi = datagen.gen_qmm(datagen.workload_seed("mlp_up"), 16, K, N, bits, group)
    ui = datagen.gen_qmm(datagen.workload_seed("mlp_up") + 100, 16, K, N, bits, group)
    x = torch.from_numpy(gi.x.view(np.int16)).to(dev).view(torch.bfloat16)
    dev_w = lambda a: (torch.from_numpy(a.words[0].view(np.int32)).to(dev),
                       torch.from_numpy(a.scales[0].view(np.int16)).to(dev).view(torch.float16),
                       torch.from_numpy(a.biases[0].view(np.int16)).to(dev).view(torch.float16))
    g0, u0 = dev_w(gi), dev_w(ui)
    del gi, ui
    copies = 4
    GS = [g0] + [tuple(t.clone() for t in g0) for _ in range(copies - 1)]
    US = [u0] + [tuple(t.clone() for t in u0) for _ in range(copies - 1)]
    plan = q.Plan(K, N, bits, group, max_M=16, out_dtype="bf16", splits=0, max_banks=2, device=dev)
    fused_row = {}
    for M in range(1, 17):
        out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        tmp = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        res = {}
        for mode in ("fused", "separate"):
            def step():
                for c in range(copies):
                    if mode == "fused":
                        q.forward_swiglu(plan, x[:M], *GS[c], *US[c], out, stream=stream)
                    else:
                        q.forward(plan, x[:M], *GS[c], tmp, stream=stream)
                        q.forward(plan, x[:M], *US[c], out, stream=stream)
            with torch.cuda.stream(stream):
                for _ in range(3):
                    step()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step()
            reps = 50
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                g.replay()
                e0.record(stream)
                for _ in range(reps):
                    g.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            res[mode] = e0.elapsed_time(e1) * 1e3 / (reps * copies)
            del g
        fused_row[str(M)] = {"fused_us": round(res["fused"], 3), "two_calls_us": round(res["separate"], 3)}
    assert plan.error_flags() == 0
    table["mlp_gate_up_swiglu:4-bit"] = {"K": K, "N": N, "group": group, "splits": plan.info()["splits"],
                                         "copies": copies, "per_M": fused_row}
    print(json.dumps({"cost_table": table, "unit": "us/call", "launch": "cuda_graph", "out": "bf16"}))


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["qmm", "reference"], default="qmm")
    ap.add_argument("--no-graph", action="store_true", help="time direct launches instead of CUDA graph replay")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-configuration timings (pr1_ref, down_longk, mixed_widths, banked)")
    ap.add_argument("--ncu-case", type=int, default=0, metavar="M",
                    help="run a small untimed profiling case with M rows and exit")
    ap.add_argument("--case-workload", default=WORKLOAD, choices=sorted(datagen.WORKLOADS))
    ap.add_argument("--case-bits", type=int, default=0)
    ap.add_argument("--case-splits", type=int, default=0)
    ap.add_argument("--calls", type=int, default=5)
    ap.add_argument("--cost-table", action="store_true",
                    help="print the per-M (1..16) us/call table of the named workloads and exit")
    args = ap.parse_args()
    if args.cost_table:
        run_cost_table(args)
        return
    if args.ncu_case:
        run_ncu_case(args)
        return
    ws, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, ws, rank)
        return
    run_gpu(args, ws, rank, local)


if __name__ == "__main__":
    main()
