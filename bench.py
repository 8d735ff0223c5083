#!/usr/bin/env python3
"""Benchmark of the CQ hot path on GB300.

One JSON line on rank 0. The headline step is the Needle-shaped decode step
(batch 1): 27 layers x {Q 512x512, K 256x512, V 256x512, gate 512x512,
O 512x512} in CQ2 plus the 8192x512 CQ4 head -- 136 matrices, 9,682,944
packed bytes -- run as ONE grouped GEMV launch over int8 per-token
activations. ``value`` is the effective GEMV bandwidth on packed bytes
(GB/s). The same run also times, each under its own events:
  * the grouped GEMM (prefill) over the same matrix set at M=2048 (TFLOP/s),
  * the encoder on 16 fp32 matrices of 8192x8192 with 1% outliers (GB/s).

L2: every config's weights fit in the 126 MB L2, so the decode step cycles
through R copies of the weight set whose footprint is >= 4x L2; each step
reads a copy that was evicted long ago.

``--impl reference`` times the oracle (plain C, fp64, single thread) on the
host cores on a bounded sample of the same workload.
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

METRIC = "CQ2 GEMV effective GB/s and % HBM roofline; CQ GEMM TOPS at M=2048"
WORKLOAD = ("Needle-shaped decode step, batch 1: 27 x {Q 512x512, K 256x512, V 256x512, gate 512x512, "
            "O 512x512} CQ2 + head 8192x512 CQ4, int8 per-token activations")

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch of a
# kernel, from one ncu capture of the bench workload, keyed by kernel and by a
# hash of the sources it was built from: once a source changes the entry no
# longer matches and traffic reads null.
NCU_TRAFFIC = {
    "gemv_fast": ("75d08df624551252", 9777664),
    "gemm_x8": ("dd123d837be7b655", 527848448),
    "encode_cq2": ("d6aa9d34094c044f", 282315008),
    "gather_cq4": ("5fb8fc86d8fb3ba1", 75002880),
    "kv_attend": ("b470d32ba9762b74", 148856064),
}
KERNEL_SOURCES = {
    "gemv_fast": ("cq_gemv_fast.cu", "cq_internal.h"),
    "gemm_x8": ("cq_gemm.cu", "cq_internal.h"),
    "encode_cq2": ("cq_encode.cu", "cq_internal.h"),
    "gather_cq4": ("cq_gather.cu", "cq_internal.h"),
    "kv_attend": ("cq_kv.cu", "cq_internal.h"),
}


def _src_hash(*names: str) -> str:
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "hadamard_rotated_codebook_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str):
    rec = NCU_TRAFFIC.get(kernel)
    if rec and rec[0] == _src_hash(*KERNEL_SOURCES[kernel]):
        return rec[1]
    return None


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str, period_ms: int = 50):
        self.cmd = ["nvidia-smi", f"--id={gpu_id}", "--query-gpu=" + ",".join(self.FIELDS),
                    "--format=csv,noheader,nounits", f"-lms={period_ms}"]
        self.rows, self.proc, self.th = [], None, None

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.th = threading.Thread(target=self._read, daemon=True)
        self.th.start()
        time.sleep(0.3)  # let the first sample land before the timed region

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == len(self.FIELDS):
                self.rows.append(parts)

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.th:
            self.th.join(timeout=5)

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            try:
                sm.append(float(r[0]))
                smax.append(float(r[1]))
            except ValueError:
                continue
            for nm, v in zip(names, r[4:]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------- workloads

def decode_workload(C, S, device, copies_min_bytes):
    import torch
    mats = S.decode_step_mats()
    cbs = {b: C.cq_codebook_init(b) for b in (2, 4)}
    sizes = [C.cq_packed_bytes(m.out, m.n_in, 128, m.bits) for m in mats]
    offs, tot = [], 0
    for sz in sizes:
        offs.append(tot)
        tot += (sz + 255) // 256 * 256
    base = torch.empty(tot, dtype=torch.uint8, device=device)
    for m, o, sz in zip(mats, offs, sizes):
        W = S.decode_weights(m, device=device)
        C.cq_encode(W, m.bits, cbs[m.bits], blob=base[o:o + sz])
    packed = sum(sizes)
    R = max(2, math.ceil(copies_min_bytes / packed))
    copies = [base] + [base.clone() for _ in range(R - 1)]
    nact = S.n_activations(mats)
    X = torch.cat([S.decode_activation(a, device=device) for a in range(nact)])  # [55, 512]
    Xq0, xs0 = C.cq_act_quant_int8(X)
    # the step's inputs in one contiguous buffer (int8 codes, then the fp32
    # scales 16-byte aligned), so that one host->device copy carries them
    xs_off = (Xq0.numel() + 15) // 16 * 16
    inbuf = torch.zeros(xs_off + 4 * xs0.numel(), dtype=torch.uint8, device=device)
    Xq = inbuf[:Xq0.numel()].view(torch.int8).view(Xq0.shape)
    xs = inbuf[xs_off:].view(torch.float32)
    Xq.copy_(Xq0)
    xs.copy_(xs0)
    out_total = sum(m.out for m in mats)
    ybuf = torch.empty(out_total, dtype=torch.float32, device=device)
    yoffs, t = [], 0
    for m in mats:
        yoffs.append(t)
        t += m.out
    wl = dict(mats=mats, R=R, packed=packed, Xq=Xq, xs=xs, inbuf=inbuf, ybuf=ybuf, copies=copies, offs=offs,
              sizes=sizes, cbs=cbs, out_total=out_total, yoffs=yoffs, xs_off=xs_off)
    wl["plans"] = make_plans(C, wl, Xq, xs, ybuf)
    wl["algo_bytes"] = packed + Xq.numel() + 4 * xs.numel() + 4 * out_total
    return wl


def make_plans(C, wl, Xq, xs, ybuf):
    """One grouped-GEMV plan per weight copy, reading the activations Xq/xs
    and writing ybuf (device tensors, or pinned host tensors)."""
    plans = []
    for cp in wl["copies"]:
        items = []
        for m, o, sz, yo in zip(wl["mats"], wl["offs"], wl["sizes"], wl["yoffs"]):
            items.append(dict(blob=cp[o:o + sz], out=m.out, **{"in": m.n_in}, bits=m.bits, codebook=wl["cbs"][m.bits],
                              x=Xq[m.act:m.act + 1], x_scale=xs[m.act:m.act + 1],
                              y=ybuf[yo:yo + m.out].view(1, m.out)))
        plans.append(C.GemvPlan(items))
    return plans


# ------------------------------------------------------------ ranks
# One process per GPU; every rank runs the whole workload on its own GPU (the
# units are independent: weak scaling, no data-path collective). Only the
# barriers around the timed region and the max of the ranks' times cross.

def rank_context():
    """(world size, rank, local rank) from the launcher's environment."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_ops(world, device):
    """barrier() and max_over_ranks(v) for an initialised process group
    (tensors on `device`: a GPU for NCCL, the CPU for gloo)."""
    import torch
    import torch.distributed as dist

    def barrier():
        if world > 1:
            dist.barrier()

    def max_over_ranks(v):
        if world == 1:
            return v
        t = torch.tensor([v], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    return barrier, max_over_ranks


def aggregate_gbs(bytes_per_rank_step, steps, world, max_ms):
    """Whole-job throughput: the bytes every rank processed over the slowest
    rank's time."""
    return world * bytes_per_rank_step * steps / (max_ms * 1e-3) / 1e9


def run_cq(args):
    import torch
    import torch.distributed as dist

    import hadamard_rotated_codebook_gb300 as C
    import synthetic as S

    world, rank, local = rank_context()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(device)
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20)
    peaks, peak_kind = measured_peaks()
    barrier, max_over_ranks = rank_ops(world, device)

    if args.only in ("gemm", "encode", "gather", "kv", "g64"):
        # one part alone, for profiling: only that part's buffers are held
        stream = torch.cuda.Stream(device)
        if args.only == "gemm":
            wl = decode_workload(C, S, device, 0)
            res = bench_gemm(C, S, torch, wl, device, stream, peaks, peak_kind, barrier, max_over_ranks, world)
        elif args.only == "gather":
            res = bench_gather(C, S, torch, device, stream, peaks, barrier, max_over_ranks, world)
        elif args.only == "kv":
            res = bench_kv(C, S, torch, device, stream, peaks, barrier, max_over_ranks, world)
        elif args.only == "g64":
            res = bench_g64(C, S, torch, device, stream, peaks, barrier, max_over_ranks, world)
        else:
            res = bench_encode(C, S, torch, device, stream, peaks, barrier, max_over_ranks, world, args.encode_count)
        if rank == 0:
            print(json.dumps(res), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return

    wl = decode_workload(C, S, device, 4 * l2)
    plans, R = wl["plans"], wl["R"]
    K, Wm = args.steps, args.warmup
    stream = torch.cuda.Stream(device)

    # ---- warm-up: W untimed steps ----
    with torch.cuda.stream(stream):
        for i in range(Wm):
            plans[i % R].run(stream)
    stream.synchronize()

    # ---- graph of `chunk` steps cycling through the copies ----
    chunk = min(K, 4 * R * max(1, 1000 // (4 * R)))
    while K % chunk:
        chunk -= 1

    def steps(n):
        for i in range(n):
            plans[i % R].run(stream)

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        steps(chunk)
    with torch.cuda.stream(stream):
        g.replay()  # upload the graph (untimed)
    stream.synchronize()

    gpu_id = f"GPU-{props.uuid}" if hasattr(props, "uuid") else str(local)
    clocks = ClockSampler(gpu_id)
    clocks.start()
    barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):  # replay() launches on the current stream
        ev0.record(stream)
        for _ in range(K // chunk):
            g.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clocks.stop()
    C.cq_device_status(device)
    ms = max_over_ranks(ev0.elapsed_time(ev1))
    ms_step = ms / K
    gbs = aggregate_gbs(wl["packed"], K, world, ms)
    launches = K  # one grouped GEMV launch per step
    achieved = wl["algo_bytes"] / (ms_step * 1e-3) / 1e9
    roofline = {
        "bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
        "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_source": peak_kind,
        "traffic": ncu_traffic("gemv_fast"),
        "kernel": "gemv (grouped decode step)",
        "algorithmic_bytes_per_launch": wl["algo_bytes"],
    }

    result = {
        "metric": METRIC, "value": round(gbs, 1), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": Wm, "ms_per_step": round(ms_step, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "matrices": len(wl["mats"]), "packed_bytes": wl["packed"],
                   "batch": 1, "weight_copies": R, "l2": f"inputs larger than L2: {R} rotating weight copies "
                   f"({R * wl['packed'] / 1e6:.0f} MB >= 4x L2 {l2 / 1e6:.0f} MB)",
                   "parallelism": f"replica x{world}" if world > 1 else "single GPU"},
        "roofline": roofline,
        "pct_of_8tbs": round(100 * (wl["packed"] * K / (ms * 1e-3) / 1e9) / 8000.0, 2),
        "gpu_launches": launches,
        "clocks": clocks.summary(),
    }

    # ---- end to end: the activations come from pinned host memory and the
    # outputs go back to pinned host memory, every step. The kernels read and
    # write those buffers in place across the host link (Grace-Blackwell
    # NVLink-C2C), the path a caller holding host buffers takes with this
    # library; a copy-engine transfer on each side measured slower here ----
    in_h = wl["inbuf"].cpu().pin_memory()
    xq_h = in_h[:wl["Xq"].numel()].view(torch.int8).view(wl["Xq"].shape)
    xs_h = in_h[wl["xs_off"]:].view(torch.float32)
    y_h = torch.zeros(wl["out_total"], dtype=torch.float32).pin_memory()
    plans_h = make_plans(C, wl, xq_h, xs_h, y_h)
    Ke = min(K, 20000)
    ce = min(chunk, Ke)
    while Ke % ce:
        ce -= 1

    def e2e_steps(n):
        for i in range(n):
            plans_h[i % R].run(stream)

    ge = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ge, stream=stream):
        e2e_steps(ce)
    with torch.cuda.stream(stream):
        ge.replay()
    stream.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(Ke // ce):
            ge.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    mse = max_over_ranks(e0.elapsed_time(e1))
    # the host-side result is the device-side one
    if not torch.equal(y_h, wl["ybuf"].cpu()):
        raise RuntimeError("end-to-end outputs differ from the device-resident run")
    result["e2e"] = {"value": round(aggregate_gbs(wl["packed"], Ke, world, mse), 1), "unit": "GB/s",
                     "h2d_bytes_per_step": wl["inbuf"].numel(),
                     "d2h_bytes_per_step": 4 * wl["out_total"], "steps": Ke,
                     "ms_per_step": round(mse / Ke, 6)}

    if not args.skip_extra:
        result["gemm"] = bench_gemm(C, S, torch, wl, device, stream, peaks, peak_kind, barrier, max_over_ranks, world)
        result["encode"] = bench_encode(C, S, torch, device, stream, peaks, barrier, max_over_ranks, world,
                                        args.encode_count)
        result["gather"] = bench_gather(C, S, torch, device, stream, peaks, barrier, max_over_ranks, world)
        result["kv"] = bench_kv(C, S, torch, device, stream, peaks, barrier, max_over_ranks, world)
        result["group64_binary"] = bench_g64(C, S, torch, device, stream, peaks, barrier, max_over_ranks, world)
    if rank == 0 and world == 1 and not args.skip_cpu:
        result["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_seconds)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.destroy_process_group()


def bench_gemm(C, S, torch, wl, device, stream, peaks, peak_kind, barrier, max_over_ranks, world, M=2048):
    mats = wl["mats"]
    nact = S.n_activations(mats)
    acts = []
    for a in range(nact):
        X = S.decode_activation(a, tokens=M, device=device)
        acts.append(C.cq_act_quant_int8(X))
    items = []
    for m, o, sz in zip(mats, wl["offs"], wl["sizes"]):
        items.append(dict(blob=wl["copies"][0][o:o + sz], out=m.out, **{"in": m.n_in}, bits=m.bits,
                          codebook=wl["cbs"][m.bits], Xq=acts[m.act][0], x_scale=acts[m.act][1],
                          Y=torch.empty((M, m.out), dtype=torch.float32, device=device)))
    flops = 2.0 * M * sum(m.out * m.n_in for m in mats)
    with torch.cuda.stream(stream):
        for _ in range(3):  # warm-up
            C.cq_gemm_grouped(items)
    stream.synchronize()
    # one prefill step (every matrix's GEMM: one persistent launch) as a graph, so
    # the host's tensor-map encoding stays outside the timed region
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        C.cq_gemm_grouped(items)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
    stream.synchronize()
    Kg = 20
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(Kg):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1)) / Kg
    C.cq_device_status(device)
    tflops = flops / (ms * 1e-3) / 1e12
    out_bytes = 4.0 * M * sum(m.out for m in mats)
    # algorithmic bytes: fp32 Y written once, each int8 activation and every
    # blob (codes + norms) read once
    act_in = {m.act: m.n_in for m in mats}
    in_bytes = float(sum(M * n for n in act_in.values()) + sum(wl["sizes"]))
    alg_bytes = out_bytes + in_bytes
    gbs = alg_bytes / (ms * 1e-3) / 1e9
    # At K = 512 with fp32 outputs the step needs more time at HBM speed
    # (alg_bytes / hbm) than at tensor speed (flops / bf16 peak): it is bound
    # by HBM; the tensor-core view is reported beside it.
    return {"metric": "CQ GEMM TFLOP/s at M=2048 (Needle-shaped matrix set, int8 per-token activations)",
            "value": round(world * tflops, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 4), "steps": Kg,
            "warmup": 3, "M": M, "l2": "outputs larger than L2 (fp32 Y, 520 MB per step)", "flops_per_step": flops,
            "output_bytes_per_step": out_bytes, "algorithmic_bytes_per_step": alg_bytes,
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4), "peak_source": peak_kind,
                         "traffic": ncu_traffic("gemm_x8"), "kernel": "gemm_x8_kernel (one launch per step)"},
            "tensor_view": {"achieved": round(tflops, 2), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                            "frac": round(tflops / peaks["bf16_tflops"], 4),
                            "peak_source": peak_kind + " (bf16 dense; fp16 operands run at the same rate)"}}


def bench_encode(C, S, torch, device, stream, peaks, barrier, max_over_ranks, world, count=0):
    n = count or S.ENCODE_COUNT
    Ws = [S.encode_matrix(i, device=device) for i in range(n)]
    cb = C.cq_codebook_init(2)
    nb = C.cq_packed_bytes(*S.ENCODE_SHAPE, 128, 2)
    blobs = [torch.empty(nb, dtype=torch.uint8, device=device) for _ in range(n)]

    def one_pass():
        for W, b in zip(Ws, blobs):
            C.cq_encode(W, 2, cb, blob=b)

    with torch.cuda.stream(stream):
        one_pass()
    stream.synchronize()
    # the pass as a graph: host-side argument checks stay out of the timed region
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        one_pass()
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    Ke = 3
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(Ke):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1)) / Ke
    elems = n * S.ENCODE_SHAPE[0] * S.ENCODE_SHAPE[1]
    algo = elems * 4 + n * nb
    gbs = algo / (ms * 1e-3) / 1e9
    return {"metric": f"CQ2 encode GB/s ({n} fp32 8192x8192 with 1% outliers -> codes + fp16 norms)",
            "value": round(world * gbs, 1), "unit": "GB/s", "ms_per_step": round(ms, 3), "steps": Ke,
            "warmup": 1, "launches_per_step": n,
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4), "traffic": ncu_traffic("encode_cq2"),
                         "algorithmic_bytes_per_launch": algo // n}}


def bench_gather(C, S, torch, device, stream, peaks, barrier, max_over_ranks, world, n=65536):
    """Row-gather dequantisation: n random token ids into the tied 8192 x 512
    CQ4 embedding/logit table of the Needle-shaped set (fp32 rows out)."""
    out, n_in = 8192, 512
    cb = C.cq_codebook_init(4)
    nb = C.cq_packed_bytes(out, n_in, 128, 4)
    blob = torch.from_numpy(S.random_blob(out * n_in * 4 // 8, out * (n_in // 128), 74)).to(device)
    assert blob.numel() == nb
    g_ = torch.Generator(device="cpu").manual_seed(75)
    idx = torch.randint(0, out, (n,), generator=g_, dtype=torch.int32).to(device)
    dst = torch.empty((n, n_in), dtype=torch.float32, device=device)
    with torch.cuda.stream(stream):
        C.cq_gather_rows(blob, out, n_in, 4, cb, idx, dst=dst)
    stream.synchronize()
    C.cq_device_status(device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        C.cq_gather_rows(blob, out, n_in, 4, cb, idx, dst=dst)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
    stream.synchronize()
    Kg = 20
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(Kg):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1)) / Kg
    C.cq_device_status(device)
    # algorithmic bytes: each indexed row's codes and norms read, its fp32 row
    # written, the indices read
    row_bytes = nb // out
    algo = n * (row_bytes + 4 * n_in + 4)
    gbs = algo / (ms * 1e-3) / 1e9
    return {"metric": f"CQ4 row gather GB/s ({n} token ids into the 8192x512 embedding table -> fp32 rows)",
            "value": round(world * gbs, 1), "unit": "GB/s", "ms_per_step": round(ms, 4), "steps": Kg,
            "warmup": 3, "l2": "outputs larger than L2 (128 MB per step)",
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4), "traffic": ncu_traffic("gather_cq4"),
                         "algorithmic_bytes_per_launch": algo}}


def bench_kv(C, S, torch, device, stream, peaks, barrier, max_over_ranks, world):
    """Decode-step attention over CQ KV caches: 256 sequences x 8192 cached
    tokens in the Needle 3 attention geometry, CQ2 keys and values, one call
    per step. Two copies of the caches (different seeds) alternate between
    steps, so a step's 144 MB never sit in L2 from the step before."""
    g = S.KV_GEOM
    Hq, Hkv, dk, dv = g["n_q_heads"], g["n_kv_heads"], g["head_dim_k"], g["head_dim_v"]
    T, nseq, bits = S.KV_TOKENS, S.KV_SEQS, S.KV_BITS
    cb = C.cq_codebook_init(bits)
    scale = 1.0 / math.sqrt(dk)
    sets = []
    for r in range(2):
        items = []
        for i in range(nseq):
            kc = torch.from_numpy(S.kv_cache_blob(T, Hkv * dk, bits, 20000 * r + 5000 + i)).to(device)
            vc = torch.from_numpy(S.kv_cache_blob(T, Hkv * dv, bits, 20000 * r + 6000 + i)).to(device)
            q = S.normal((Hq, dk), 20000 * r + 7000 + i).to(device)
            items.append(dict(k_cache=kc, v_cache=vc, cap=T, n_tokens=T, q=q,
                              o=torch.empty((Hq, dv), dtype=torch.float32, device=device)))
        sets.append(items)
    with torch.cuda.stream(stream):  # grows the workspace before capture
        for items in sets:
            C.cq_kv_attend(items, Hq, Hkv, dk, dv, bits, bits, cb, cb, scale)
    stream.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=stream):
        for items in sets:
            C.cq_kv_attend(items, Hq, Hkv, dk, dv, bits, bits, cb, cb, scale)
    with torch.cuda.stream(stream):
        for _ in range(3):
            gr.replay()
    stream.synchronize()
    Kg = 20
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(Kg):
            gr.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1)) / (2 * Kg)
    # algorithmic bytes: every attended cache row's codes and norms, the
    # queries read and the outputs written
    kb = C.cq_packed_bytes(T, Hkv * dk, 128, bits)
    vb = C.cq_packed_bytes(T, Hkv * dv, 128, bits)
    algo = nseq * (kb + vb + 4 * Hq * dk + 4 * Hq * dv)
    gbs = algo / (ms * 1e-3) / 1e9
    tok = nseq * T / (ms * 1e-3)
    return {"metric": f"CQ{bits} KV-cache decode attention GB/s ({nseq} sequences x {T} tokens, "
                      f"{Hq} query heads of {dk} over {Hkv} KV heads, values of {dv})",
            "value": round(world * gbs, 1), "unit": "GB/s", "ms_per_step": round(ms, 4),
            "cached_tokens_per_s": round(world * tok, 1), "steps": 2 * Kg, "warmup": 6,
            "l2": "two cache copies alternate (288 MB cycle, 2.2x L2)",
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4), "traffic": ncu_traffic("kv_attend"),
                         "algorithmic_bytes_per_launch": algo}}


def bench_g64(C, S, torch, device, stream, peaks, barrier, max_over_ranks, world):
    """Group-64 CQ2 and binary (group 128) weights: one grouped GEMV launch
    over 64 matrices of 4096 x 4096 (batch 1, fp32 activations), the set
    larger than L2, plus the encoder on 4 x 8192^2 at group 64 CQ2."""
    res = {}
    for name, group, bits in (("cq2_group64", 64, 2), ("binary_group128", 128, 1), ("cq2_group128", 128, 2)):
        out = n_in = 4096
        cb = C.cq_codebook_init(bits, group)
        nb = C.cq_packed_bytes(out, n_in, group, bits)
        ip = (n_in + group - 1) // group * group
        items = []
        for i in range(64):
            blob = torch.from_numpy(S.random_blob(out * ip * (2 if bits == 5 else bits) // 8, out * ip // group,
                                                  30000 + 100 * bits + i)).to(device)
            x = S.normal((1, n_in), 31000 + i).to(device)
            items.append(dict(blob=blob, out=out, **{"in": n_in}, bits=bits, codebook=cb, x=x, group=group,
                              y=torch.empty((1, out), dtype=torch.float32, device=device)))
        plan = C.GemvPlan(items)
        with torch.cuda.stream(stream):
            for _ in range(3):
                plan.run(stream)
        stream.synchronize()
        Kg = 20
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(Kg):
                plan.run(stream)
            e1.record(stream)
        torch.cuda.synchronize()
        ms = max_over_ranks(e0.elapsed_time(e1)) / Kg
        algo = 64 * (nb + 4 * n_in + 4 * out)
        gbs = algo / (ms * 1e-3) / 1e9
        res[name] = {"metric": f"GEMV GB/s, 64 x 4096x4096, group {group}, {bits}-bit codes, batch 1",
                     "value": round(world * gbs, 1), "unit": "GB/s", "ms_per_step": round(ms, 4), "steps": Kg,
                     "packed_bytes_per_step": 64 * nb,
                     "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                  "frac": round(gbs / peaks["hbm_gbs"], 4), "traffic": None,
                                  "algorithmic_bytes_per_launch": algo}}
    # encoder at group 64
    cb = C.cq_codebook_init(2, 64)
    Ws = [S.normal((8192, 8192), 32000 + i, S.W_STD, device=device) for i in range(4)]
    blobs = [torch.empty(C.cq_packed_bytes(8192, 8192, 64, 2), dtype=torch.uint8, device=device) for _ in range(4)]
    with torch.cuda.stream(stream):
        for _ in range(3):
            C.cq_encode(Ws[0], 2, cb, group=64, blob=blobs[0])
    stream.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for W, bl in zip(Ws, blobs):
            C.cq_encode(W, 2, cb, group=64, blob=bl)
        e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1)) / 4
    algo = 8192 * 8192 * 4 + blobs[0].numel()
    gbs = algo / (ms * 1e-3) / 1e9
    res["encode_cq2_group64"] = {"metric": "encode GB/s, 8192x8192 fp32 -> CQ2 at group 64",
                                 "value": round(world * gbs, 1), "unit": "GB/s", "ms_per_matrix": round(ms, 4),
                                 "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                                              "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                                              "traffic": None, "algorithmic_bytes_per_launch": algo}}
    return res


# ------------------------------------------------------------ CPU oracle

def _oracle_step_sample(budget_s: float):
    """Times the oracle's product (dequantise with the explicit Hadamard,
    fp64 matmul) over decode-step matrices in order until `budget_s` is
    spent; returns (packed bytes processed, seconds, matrices)."""
    import numpy as np

    import oracle as O
    import synthetic as S
    mats = S.decode_step_mats()
    cbs = {b: O.analytic_codebook(b) for b in (2, 4)}
    done_bytes, t_used, n = 0, 0.0, 0
    for i, m in enumerate(mats):
        ip = O.in_padded(m.n_in)
        blob = S.random_blob(m.out * ip * O.width(m.bits) // 8, m.out * ip // 128, 9000 + i)
        x = S.decode_activation(m.act).numpy()
        q, s = O.act_quant_int8(x)
        xt = q.astype(np.float64) * s.astype(np.float64)[:, None]
        t0 = time.perf_counter()
        What = O.dequant(blob, m.out, m.n_in, m.bits, cbs[m.bits])
        O.matmul(What, xt)
        t_used += time.perf_counter() - t0
        done_bytes += blob.size
        n += 1
        if t_used >= budget_s:
            break
    return done_bytes, t_used, n


def cpu_baseline(budget_s: float = 10.0):
    b, t, n = _oracle_step_sample(budget_s)
    return {"value": round(b / t / 1e9, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"oracle dequantise + fp64 matmul over the first {n} decode-step matrices "
                      f"({b} packed bytes) in {t:.1f} s, single thread"}


def run_reference(args):
    world, rank, _ = rank_context()
    if rank != 0:  # the oracle runs on rank 0 alone; the other ranks exit without work
        return
    K, Wm = args.steps, args.warmup
    per_step = max(0.05, min(2.0, 120.0 / max(1, min(K, 200) + Wm)))
    K_run = min(K, 200)
    for _ in range(min(Wm, 3)):
        _oracle_step_sample(per_step / 4)
    tot_b, tot_t = 0, 0.0
    for _ in range(K_run):
        b, t, _ = _oracle_step_sample(per_step)
        tot_b += b
        tot_t += t
    v = tot_b / tot_t / 1e9
    res = {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "GB/s", "n_gpus": world,
           "steps": K_run, "warmup": Wm, "ms_per_step": round(1e3 * tot_t / K_run, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": WORKLOAD, "sample": f"about {per_step:.2f} s of oracle work per step"},
           "cpu_baseline": {"value": round(v, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
                            "sample": "decode-step matrices in order, oracle dequantise + fp64 matmul"},
           "e2e": {"value": round(v, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100000)
    ap.add_argument("--warmup", type=int, default=1000)
    ap.add_argument("--impl", default="cq", choices=["cq", "reference"])
    ap.add_argument("--skip-extra", action="store_true", help="decode step only")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--encode-count", type=int, default=0, help="matrices in the encode part (default 16)")
    ap.add_argument("--only", default="all", choices=["all", "gemm", "encode", "gather", "kv", "g64"],
                    help="time one secondary part alone and print its JSON object (profiling)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_cq(args)


if __name__ == "__main__":
    main()
