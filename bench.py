#!/usr/bin/env python3
"""Benchmark of the CQ hot path on GB300.

One JSON line on rank 0. The headline step is the Needle-shaped decode step
(batch 1): 27 layers x {Q 512x512, K 256x512, V 256x512, gate 512x512,
O 512x512} in CQ2 plus the 8192x512 CQ4 head -- 136 matrices, 9,682,944
packed bytes -- run as ONE grouped GEMV launch over int8 per-token
activations. ``value`` is the effective GEMV bandwidth on packed bytes
(GB/s). The same run also times, each under its own events:
  * the single 512x512 CQ2 matrix at batch 1,
  * the width sweep: 4096x4096 and 14336x4096 in CQ2/CQ3/CQ4/ternary at
    batch 1 and 16,
  * the grouped GEMM (prefill) over the decode-step matrix set at M = 64,
    256 and 2048 (TFLOP/s),
  * the encoder on 16 fp32 matrices of 8192x8192 with 1% outliers (GB/s),
    then the container round trip and a batch-1 GEMV over a reloaded blob,
  * the row gather, the CQ KV-cache attention, group 64 and binary codes.

L2: every timed input set is larger than 4x L2 (rotating copies of the
weights, or of the outputs where those dominate), so no step reads what an
earlier step left in L2.

Timing: CUDA events on the launching stream, behind a spin kernel so that
the host's enqueue rate stays out of the region; barrier + synchronize on
both sides; the max over ranks.

At the end, on rank 0 at N=1, the oracle leg runs the oracle on the host
cores: the CPU baseline (one thread and all cores) on the decode step's own
blobs, and the parity statistics of every timed workload from the samples
the GPU parts kept.

``--impl reference`` times the oracle (plain C, fp64, threads over row
blocks) on the host cores on a bounded sample of the same workload.
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
    "gemv_fast": ("c065cae4293b496e", 9777920),
    "gemm_x8": ("d0a5df649171482d", 527082496),
    "encode_cq2": ("c54b6c53364c8e02", 281818368),
    "gather_cq4": ("0390d90ce5f9910f", 74095616),
    "kv_attend": ("0da1ac7053c1367e", 148571392),
    "gemv_split": ("685314efe7f000a8", 289836288),
    "gemv_split_g64": ("685314efe7f000a8", 306625536),
}
KERNEL_SOURCES = {
    "gemv_fast": ("cq_gemv_fast.cu", "cq_internal.h"),
    "gemm_x8": ("cq_gemm.cu", "cq_internal.h"),
    "encode_cq2": ("cq_encode.cu", "cq_internal.h"),
    "gather_cq4": ("cq_gather.cu", "cq_internal.h"),
    "kv_attend": ("cq_kv.cu", "cq_internal.h"),
    "gemv_split": ("cq_gemv_wide.cu", "cq_internal.h"),
    "gemv_split_g64": ("cq_gemv_wide.cu", "cq_internal.h"),
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


# ---------------------------------------------------------------- timing

def sleep_cycles(replays: int) -> int:
    """Cycles of the spin kernel that precedes a timed region: long enough
    for the host to enqueue the region's launches behind it, so that the
    events time the device work and not the host's enqueue rate."""
    return 4_000_000 + 60_000 * replays


def timed(torch, stream, fn, replays, barrier, max_over_ranks):
    """Milliseconds of `replays` calls of fn() on `stream`, timed with CUDA
    events on that stream: barrier and synchronize on both sides; a spin
    kernel before the first event keeps host enqueue time out of the region."""
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(sleep_cycles(replays))
        e0.record(stream)
        for _ in range(replays):
            fn()
        e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    return max_over_ranks(e0.elapsed_time(e1))


def graph_of(torch, stream, fn):
    """fn() captured as a CUDA graph on `stream` (replayed once, untimed, to
    upload it)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    return g


def copies_for(nbytes: int, l2: int) -> int:
    """Rotating copies of an input of `nbytes` whose footprint is >= 4x L2."""
    return max(2, math.ceil(4 * l2 / max(1, nbytes)))


def hbm_roofline(gbs, peaks, peak_kind, traffic=None, **extra):
    r = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
         "frac": round(gbs / peaks["hbm_gbs"], 4), "peak_source": peak_kind, "traffic": traffic}
    r.update(extra)
    return r


# ------------------------------------------------------ parity samples
# The GPU parts keep sampled inputs and outputs of the workloads they time
# (host copies, taken after their timed regions); the oracle leg at the end
# of the run recomputes those outputs with the oracle and reports the
# comparison. Nothing here runs the oracle.

class Samples:
    def __init__(self):
        self.items = []

    def add(self, path, kind, **data):
        self.items.append(dict(path=tuple(path), kind=kind, **data))


def sample_rows(out: int, k: int) -> "np.ndarray":
    import numpy as np
    if out <= k:
        return np.arange(out)
    r = np.unique(np.linspace(0, out - 1, k).round().astype(np.int64))
    return r


def host_sub_blob(blob_np, out, n_in, bits, rows, group=128):
    """Blob of a subset of rows (their code rows, then their norms)."""
    import numpy as np
    ip = (n_in + group - 1) // group * group
    w = 2 if bits == 5 else bits
    rb = ip * w // 8
    ng = ip // group
    codes = blob_np[: out * rb].reshape(out, rb)[rows]
    norms = blob_np[out * rb:].reshape(out, ng * 2)[rows]
    return np.concatenate([codes.ravel(), norms.ravel()])


# ------------------------------------------------------------- workloads

def decode_workload(C, S, device, copies_min_bytes, samples=None):
    import numpy as np
    import torch
    mats = S.decode_step_mats()
    cbs = {b: C.cq_codebook_init(b) for b in (2, 4)}
    sizes = [C.cq_packed_bytes(m.out, m.n_in, 128, m.bits) for m in mats]
    offs, tot = [], 0
    for sz in sizes:
        offs.append(tot)
        tot += (sz + 255) // 256 * 256
    base = torch.empty(tot, dtype=torch.uint8, device=device)
    w_rows = []
    for m, o, sz in zip(mats, offs, sizes):
        W = S.decode_weights(m, device=device)
        C.cq_encode(W, m.bits, cbs[m.bits], blob=base[o:o + sz])
        rows = sample_rows(m.out, 4)
        w_rows.append((rows, W[torch.from_numpy(rows).to(device)].cpu().numpy()))
    packed = sum(sizes)
    R = max(2, math.ceil(copies_min_bytes / packed))
    copies = [base] + [base.clone() for _ in range(R - 1)]
    nact = S.n_activations(mats)
    X = torch.cat([S.decode_activation(a, device=device) for a in range(nact)])  # [55, 512] fp32
    Xq0, xs0 = C.cq_act_quant_int8(X)
    # the step's inputs in one contiguous buffer (int8 codes, then the fp32
    # scales 16-byte aligned)
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
    wl = dict(mats=mats, R=R, packed=packed, X=X, Xq=Xq, xs=xs, inbuf=inbuf, ybuf=ybuf, copies=copies, offs=offs,
              sizes=sizes, cbs=cbs, out_total=out_total, yoffs=yoffs, xs_off=xs_off, w_rows=w_rows)
    wl["plans"] = make_plans(C, wl, Xq, xs, ybuf)
    wl["algo_bytes"] = packed + Xq.numel() + 4 * xs.numel() + 4 * out_total
    return wl


def make_plans(C, wl, Xq, xs, ybuf):
    """One grouped-GEMV plan per weight copy, reading the activations Xq/xs
    and writing ybuf (device tensors, or pinned host tensors). With xs None,
    Xq holds fp32 activations that the call quantises per token itself."""
    plans = []
    for cp in wl["copies"]:
        items = []
        for m, o, sz, yo in zip(wl["mats"], wl["offs"], wl["sizes"], wl["yoffs"]):
            act = (dict(x=Xq[m.act:m.act + 1], quantize=True) if xs is None else
                   dict(x=Xq[m.act:m.act + 1], x_scale=xs[m.act:m.act + 1]))
            items.append(dict(blob=cp[o:o + sz], out=m.out, **{"in": m.n_in}, bits=m.bits, codebook=wl["cbs"][m.bits],
                              y=ybuf[yo:yo + m.out].view(1, m.out), **act))
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


class Ctx:
    """What every part of the run shares."""

    def __init__(self, C, S, torch, device, stream, peaks, peak_kind, barrier, max_over_ranks, world, l2, samples):
        self.C, self.S, self.torch, self.device, self.stream = C, S, torch, device, stream
        self.peaks, self.peak_kind = peaks, peak_kind
        self.barrier, self.max_over_ranks, self.world, self.l2 = barrier, max_over_ranks, world, l2
        self.samples = samples

    def timed(self, fn, replays):
        return timed(self.torch, self.stream, fn, replays, self.barrier, self.max_over_ranks)


def run_cq(args):
    import numpy as np
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
    stream = torch.cuda.Stream(device)
    samples = Samples()
    cx = Ctx(C, S, torch, device, stream, peaks, peak_kind, barrier, max_over_ranks, world, l2, samples)

    if args.only != "all":
        # one part alone, for profiling: only that part's buffers are held
        if args.only == "gemm":
            wl = decode_workload(C, S, device, 0)
            res = bench_gemm(cx, wl, 2048)
        elif args.only == "gemm_small":
            wl = decode_workload(C, S, device, 0)
            res = {f"m{M}": bench_gemm(cx, wl, M) for M in (64, 256)}
        elif args.only == "gather":
            res = bench_gather(cx)
        elif args.only == "kv":
            res = bench_kv(cx)
        elif args.only == "g64":
            res = bench_g64(cx)
        elif args.only == "sweep":
            res = bench_sweep(cx)
        elif args.only == "single":
            res = bench_single(cx)
        elif args.only == "decode":
            wl = decode_workload(C, S, device, 4 * l2)
            res = bench_decode(cx, wl, args.steps, args.warmup)
        else:
            res = bench_encode(cx, args.encode_count)
        if rank == 0:
            print(json.dumps(res), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return

    wl = decode_workload(C, S, device, 4 * l2, samples)
    gpu_id = f"GPU-{props.uuid}" if hasattr(props, "uuid") else str(local)
    clocks = ClockSampler(gpu_id)
    clocks.start()
    dec = bench_decode(cx, wl, args.steps, args.warmup)
    clocks.stop()
    C.cq_device_status(device)
    ms = dec["ms"]
    K = args.steps
    ms_step = ms / K
    gbs = aggregate_gbs(wl["packed"], K, world, ms)
    achieved = wl["algo_bytes"] / (ms_step * 1e-3) / 1e9
    result = {
        "metric": METRIC, "value": round(gbs, 1), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "matrices": len(wl["mats"]), "packed_bytes": wl["packed"],
                   "batch": 1, "weight_copies": wl["R"], "l2": f"inputs larger than L2: {wl['R']} rotating weight "
                   f"copies ({wl['R'] * wl['packed'] / 1e6:.0f} MB >= 4x L2 {l2 / 1e6:.0f} MB)",
                   "timing": "CUDA events on the launching stream around K graph-captured steps, "
                             "behind a spin kernel that keeps host enqueue time out of the region",
                   "parallelism": f"replica x{world}" if world > 1 else "single GPU"},
        "roofline": hbm_roofline(achieved, peaks, peak_kind, ncu_traffic("gemv_fast"),
                                 kernel="gemv_fast_kernel (grouped decode step, one launch per step)",
                                 algorithmic_bytes_per_launch=wl["algo_bytes"]),
        "pct_of_8tbs": round(100 * gbs / world / 8000.0, 2),
        "gpu_launches": K,  # one grouped GEMV launch per step
        "clocks": clocks.summary(),
    }
    # parity sample of the decode step: every matrix's outputs of the last
    # timed step, its blob and its activation (the oracle leg recomputes them)
    base_np = wl["copies"][0].cpu().numpy()
    ybuf_np = wl["ybuf"].cpu().numpy()
    Xq_np, xs_np = wl["Xq"].cpu().numpy(), wl["xs"].cpu().numpy()
    samples.add(("parity",), "decode", wl=dict(
        mats=wl["mats"], blobs=[base_np[o:o + sz] for o, sz in zip(wl["offs"], wl["sizes"])],
        cbs=wl["cbs"], Xq=Xq_np, xs=xs_np, y=[ybuf_np[yo:yo + m.out] for m, yo in zip(wl["mats"], wl["yoffs"])],
        w_rows=wl["w_rows"]))

    result["e2e"], result["e2e_graph"] = bench_e2e(cx, wl, K)

    if not args.skip_extra:
        result["single"] = bench_single(cx)
        result["sweep"] = bench_sweep(cx)
        result["gemm"] = bench_gemm(cx, wl, 2048)
        result["gemm_small"] = {f"m{M}": bench_gemm(cx, wl, M) for M in (64, 256)}
        del wl
        result["encode"] = bench_encode(cx, args.encode_count)
        result["gather"] = bench_gather(cx)
        result["kv"] = bench_kv(cx)
        result["group64_binary"] = bench_g64(cx)
    if rank == 0 and world == 1 and not args.skip_cpu:
        oracle_leg(result, samples, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.destroy_process_group()


def bench_decode(cx, wl, K, Wm):
    """The headline: K decode steps (one grouped GEMV launch each) over the
    rotating weight copies, captured as CUDA graphs of `chunk` steps."""
    torch, stream = cx.torch, cx.stream
    plans, R = wl["plans"], wl["R"]
    with torch.cuda.stream(stream):
        for i in range(Wm):
            plans[i % R].run(stream)
    stream.synchronize()
    chunk = min(K, 4 * R * max(1, 1000 // (4 * R)))
    while K % chunk:
        chunk -= 1

    def steps():
        for i in range(chunk):
            plans[i % R].run(stream)

    g = graph_of(torch, stream, steps)
    ms = cx.timed(g.replay, K // chunk)
    return {"ms": ms, "ms_per_step": ms / K}


def bench_e2e(cx, wl, K):
    """The decode step end to end through the public API: every step copies
    its fp32 activations from pinned host memory to the device and runs the
    grouped GEMV on them with per-token int8 quantisation inside the call
    (CQ_X_F32Q: bit-identical to cq_act_quant_int8 followed by the int8
    call); its kernel writes the outputs into pinned host memory in place
    (the host link, NVLink-C2C on Grace-Blackwell), and the host waits for
    the step before the next one. `e2e` makes the calls eagerly (the ctypes calls, argument
    checks and launches are inside the region); `e2e_graph` replays the same
    calls captured once as a CUDA graph."""
    torch, C, stream, R = cx.torch, cx.C, cx.stream, wl["R"]
    X_h = wl["X"].cpu().pin_memory()
    X_d = torch.empty_like(wl["X"])
    y_h = torch.zeros(wl["out_total"], dtype=torch.float32).pin_memory()
    plans_h = make_plans(C, wl, X_d, None, y_h)
    h2d, d2h = X_h.numel() * 4, 4 * wl["out_total"]

    def one(i):
        X_d.copy_(X_h, non_blocking=True)
        plans_h[i % R].run(stream)

    Ke = min(K, 2000)
    with torch.cuda.stream(stream):
        for i in range(3):
            one(i)
    stream.synchronize()
    cnt = [0]

    def eager_step():
        one(cnt[0])
        cnt[0] += 1
        stream.synchronize()  # the host reads the step's result

    # five batches of eager steps; the host clock of a shared machine sees
    # occasional stalls of other processes, so the median batch is reported
    nb = 5
    per = max(1, Ke // nb)
    batch_ms = []
    for _ in range(nb):
        cx.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for _ in range(per):
                eager_step()
        t1 = time.perf_counter()
        cx.barrier()
        batch_ms.append(cx.max_over_ranks(1e3 * (t1 - t0)))
    Ke = per * nb
    ms = statistics.median(batch_ms) * nb
    if not torch.equal(y_h, wl["ybuf"].cpu()):
        raise RuntimeError("end-to-end outputs differ from the device-resident run")
    e2e = {"value": round(aggregate_gbs(wl["packed"], Ke, cx.world, ms), 1), "unit": "GB/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": Ke, "ms_per_step": round(ms / Ke, 6),
           "batch_ms_per_step": [round(b / per, 6) for b in batch_ms],
           "timing": f"host wall clock over eager steps, each ending in a stream synchronize; median of {nb} "
                     f"batches of {per} steps",
           "path": "fp32 activations pinned host -> device copy -> cq_gemv_grouped with per-token int8 "
                   "quantisation in the call (outputs written to pinned host memory in place)"}

    Kg = min(K, 20000)
    ce = min(Kg, 4 * R * max(1, 1000 // (4 * R)))
    while Kg % ce:
        ce -= 1

    def graph_steps():
        for i in range(ce):
            one(i)

    y_h.zero_()
    ge = graph_of(torch, stream, graph_steps)
    ms = cx.timed(ge.replay, Kg // ce)
    if not torch.equal(y_h, wl["ybuf"].cpu()):
        raise RuntimeError("graph end-to-end outputs differ from the device-resident run")
    eg = {"value": round(aggregate_gbs(wl["packed"], Kg, cx.world, ms), 1), "unit": "GB/s",
          "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": Kg, "ms_per_step": round(ms / Kg, 6),
          "gpu_launches_per_step": 1, "copies_per_step": 1,
          "timing": "CUDA events around graph replays of the same steps"}
    return e2e, eg


def gemv_line(cx, path, blob, out, n_in, bits, cb, x, group=128, xs=None, kernel=""):
    """Times one GEMV shape: the blob cloned into rotating copies (>= 4x L2),
    one call per step, steps captured as a CUDA graph cycling through the
    copies. Returns the line and stores a parity sample."""
    import numpy as np
    torch, C, stream = cx.torch, cx.C, cx.stream
    nb = blob.numel()
    # >= 4x L2 of copies; a matrix of tens of KB is capped at 2400 copies
    # (still more than L2), which keeps its graph's launch parameters small
    R = min(copies_for(nb, cx.l2), 2400)
    big = torch.empty(R * ((nb + 255) // 256 * 256), dtype=torch.uint8, device=cx.device)
    stride = (nb + 255) // 256 * 256
    views = []
    for r in range(R):
        v = big[r * stride:r * stride + nb]
        v.copy_(blob)
        views.append(v)
    B = x.shape[0]
    y = torch.empty((B, out), dtype=torch.float32, device=cx.device)
    plans = [C.GemvPlan([dict(blob=v, out=out, **{"in": n_in}, bits=bits, codebook=cb, x=x, x_scale=xs, y=y,
                              group=group)]) for v in views]
    with torch.cuda.stream(stream):
        for i in range(3):
            plans[i % R].run(stream)
    stream.synchronize()
    per_graph = R * max(1, 64 // R)

    def steps():
        for i in range(per_graph):
            plans[i % R].run(stream)

    g = graph_of(torch, stream, steps)
    reps = max(1, 256 // per_graph)
    ms = cx.timed(g.replay, reps) / (reps * per_graph)
    xbytes = x.numel() * x.element_size() + (4 * B if xs is not None else 0)
    algo = nb + xbytes + 4 * B * out
    gbs = algo / (ms * 1e-3) / 1e9
    rows = sample_rows(out, 48)
    cx.samples.add(path, "gemv", blob=host_sub_blob(blob.cpu().numpy(), out, n_in, bits, rows, group),
                   rows=rows, n_in=n_in, bits=bits, group=group, cb=np.asarray(cb),
                   x=(x.cpu().numpy().astype(np.float64) if xs is None else
                      x.cpu().numpy().astype(np.float64) * xs.cpu().numpy().astype(np.float64)[:, None]),
                   y=y.cpu().numpy()[:, rows])
    del big, views, plans, g
    return {"value": round(cx.world * gbs, 1), "unit": "GB/s", "us_per_call": round(1e3 * ms, 3),
            "packed_bytes": nb, "batch": B, "weight_copies": R,
            "l2": f"{R} rotating copies ({R * nb / 1e6:.0f} MB, {R * nb / cx.l2:.1f}x L2)",
            "roofline": hbm_roofline(gbs, cx.peaks, cx.peak_kind, None, kernel=kernel,
                                     algorithmic_bytes_per_launch=algo)}


def gemv_kernel_name(out, n_in, bits, B, group=128):
    """Which GEMV kernel the library picks for a single matrix of this shape."""
    ng = (n_in + group - 1) // group
    ng128 = (n_in + 127) // 128
    w = 2 if bits == 5 else bits
    if group == 64 and B <= 4 and n_in % 128 == 0 and w != 3 and ng128 <= 128:
        return "gemv_split_kernel"
    if B <= 4 and group == 128 and w != 3 and ng < 16:
        return "gemv_fast_kernel"
    cols = 2 * B if B <= 4 else 8 * ((B + 7) // 8)
    if group == 128 and ng <= 128 and ng * cols * 256 + B * ng * 4 <= 136 * 1024:
        if B <= 4:
            return "gemv_split_kernel"
        return "act_frag_kernel + gemv_wide_kernel"
    return "gemv_kernel (fp32)"


def bench_single(cx):
    """The single 512x512 CQ2 matrix, batch 1, fp32 activation."""
    C, S, torch = cx.C, cx.S, cx.torch
    cb = C.cq_codebook_init(2)
    W = S.single_weights(device=cx.device)
    blob = C.cq_encode(W, 2, cb)
    x = S.single_activation(device=cx.device)
    line = gemv_line(cx, ("single",), blob, 512, 512, 2, cb, x, kernel=gemv_kernel_name(512, 512, 2, 1))
    line["metric"] = "GEMV GB/s, one 512x512 CQ2 matrix, batch 1, fp32 activation"
    rows = sample_rows(512, 8)
    cx.samples.add(("single",), "encode", W=W[torch.from_numpy(rows).to(cx.device)].cpu().numpy(),
                   blob=host_sub_blob(blob.cpu().numpy(), 512, 512, 2, rows), bits=2, group=128, cb=cb)
    return line


def bench_sweep(cx):
    """Width sweep: 4096x4096 and 14336x4096 in CQ2, CQ3, CQ4 and ternary at
    batch 1 and 16, Student-t weights, fp32 activations."""
    C, S, torch = cx.C, cx.S, cx.torch
    res = {}
    for shape in S.SWEEP_SHAPES:
        out, n_in = shape
        for bits in S.SWEEP_BITS:
            cb = C.cq_codebook_init(bits)
            W = S.sweep_weights(shape, bits, device=cx.device)
            blob = C.cq_encode(W, bits, cb)
            wname = {2: "cq2", 3: "cq3", 4: "cq4", 5: "ternary"}[bits]
            rows = sample_rows(out, 6)
            cx.samples.add(("sweep", f"{out}x{n_in}_{wname}_encode"), "encode",
                           W=W[torch.from_numpy(rows).to(cx.device)].cpu().numpy(),
                           blob=host_sub_blob(blob.cpu().numpy(), out, n_in, bits, rows), bits=bits, group=128, cb=cb)
            del W
            for B in S.SWEEP_BATCHES:
                x = S.sweep_activation(B, n_in, device=cx.device)
                key = f"{out}x{n_in}_{wname}_b{B}"
                line = gemv_line(cx, ("sweep", key), blob, out, n_in, bits, cb, x, kernel=gemv_kernel_name(out, n_in, bits, B))
                line["metric"] = f"GEMV GB/s, {out}x{n_in} {wname.upper()}, batch {B}, fp32 activations"
                res[key] = line
            res[f"{out}x{n_in}_{wname}_encode"] = {"what": "encoder parity on sampled rows of the matrix above"}
    return res


def bench_gemm(cx, wl, M):
    """The grouped GEMM (prefill) over the Needle-shaped matrix set, M tokens
    of int8 activations per input, one persistent launch per step. At M=64
    and 256 the step rotates through weight copies (the weights are what it
    streams); at M=2048 the fp32 outputs (520 MB) exceed L2."""
    import numpy as np
    C, S, torch, stream = cx.C, cx.S, cx.torch, cx.stream
    mats = wl["mats"]
    nact = S.n_activations(mats)
    acts = []
    for a in range(nact):
        X = S.decode_activation(a, tokens=M, device=cx.device)
        acts.append(C.cq_act_quant_int8(X))
    Ys = [torch.empty((M, m.out), dtype=torch.float32, device=cx.device) for m in mats]
    n_copies = 1 if M >= 2048 else min(len(wl["copies"]), copies_for(wl["packed"], cx.l2))
    item_sets = []
    for cp in wl["copies"][:n_copies]:
        item_sets.append([dict(blob=cp[o:o + sz], out=m.out, **{"in": m.n_in}, bits=m.bits, codebook=wl["cbs"][m.bits],
                               Xq=acts[m.act][0], x_scale=acts[m.act][1], Y=Y)
                          for m, o, sz, Y in zip(mats, wl["offs"], wl["sizes"], Ys)])
    flops = 2.0 * M * sum(m.out * m.n_in for m in mats)
    with torch.cuda.stream(stream):
        for items in item_sets[:3] if n_copies > 1 else item_sets * 3:
            C.cq_gemm_grouped(items)
    stream.synchronize()

    def steps():
        for items in item_sets:
            C.cq_gemm_grouped(items)

    g = graph_of(torch, stream, steps)
    reps = 200 if M >= 2048 else max(1, 600 // n_copies)
    ms = cx.timed(g.replay, reps) / (reps * n_copies)
    C.cq_device_status(cx.device)
    tflops = flops / (ms * 1e-3) / 1e12
    out_bytes = 4.0 * M * sum(m.out for m in mats)
    act_in = {m.act: m.n_in for m in mats}
    in_bytes = float(sum(M * n for n in act_in.values()) + sum(wl["sizes"]) + 4 * M * len(act_in))
    alg_bytes = out_bytes + in_bytes
    gbs = alg_bytes / (ms * 1e-3) / 1e9
    # parity sample: 4 tokens x 8 rows of every matrix
    toks = sample_rows(M, 4)
    base_np = wl["copies"][0].cpu().numpy()
    per = []
    for m, o, sz, Y in zip(mats, wl["offs"], wl["sizes"], Ys):
        rows = sample_rows(m.out, 8)
        per.append(dict(blob=host_sub_blob(base_np[o:o + sz], m.out, m.n_in, m.bits, rows), rows=rows,
                        n_in=m.n_in, bits=m.bits, cb=wl["cbs"][m.bits],
                        x=(acts[m.act][0][torch.from_numpy(toks).to(cx.device)].cpu().numpy().astype(np.float64) *
                           acts[m.act][1][torch.from_numpy(toks).to(cx.device)].cpu().numpy()
                           .astype(np.float64)[:, None]),
                        y=Y[torch.from_numpy(toks).to(cx.device)][:, torch.from_numpy(rows).to(cx.device)]
                        .cpu().numpy()))
    cx.samples.add(("gemm" if M >= 2048 else "gemm_small", f"m{M}"), "gemm", per=per)
    # At K = 512 with fp32 outputs the step needs more time at HBM speed
    # (alg_bytes / hbm) than at tensor speed (flops / bf16 peak): it is bound
    # by HBM; the tensor-core view is reported beside it.
    l2note = ("outputs larger than L2 (fp32 Y, 520 MB per step)" if M >= 2048 else
              f"{n_copies} rotating weight copies ({n_copies * wl['packed'] / 1e6:.0f} MB >= 4x L2)")
    return {"metric": f"CQ GEMM TFLOP/s at M={M} (Needle-shaped matrix set, int8 per-token activations)",
            "value": round(cx.world * tflops, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 5),
            "steps": reps * n_copies, "warmup": 3, "M": M, "l2": l2note, "flops_per_step": flops,
            "output_bytes_per_step": out_bytes, "algorithmic_bytes_per_step": alg_bytes,
            "roofline": hbm_roofline(gbs, cx.peaks, cx.peak_kind, ncu_traffic("gemm_x8") if M >= 2048 else None,
                                     kernel="gemm_x8_kernel (one launch per step)"),
            "tensor_view": {"achieved": round(tflops, 2), "peak": cx.peaks["bf16_tflops"], "unit": "TFLOP/s",
                            "frac": round(tflops / cx.peaks["bf16_tflops"], 4),
                            "peak_source": cx.peak_kind + " (bf16 dense; fp16 operands run at the same rate)"}}


def bench_encode(cx, count=0):
    """The encoder on 16 fp32 8192x8192 matrices with 1% outliers, then the
    container round trip of the 16 blobs and a batch-1 GEMV over one
    reloaded blob (fed to the kernel as read)."""
    import tempfile

    import numpy as np
    C, S, torch, stream = cx.C, cx.S, cx.torch, cx.stream
    n = count or S.ENCODE_COUNT
    out, n_in = S.ENCODE_SHAPE
    Ws = [S.encode_matrix(i, device=cx.device) for i in range(n)]
    cb = C.cq_codebook_init(2)
    nb = C.cq_packed_bytes(out, n_in, 128, 2)
    blobs = [torch.empty(nb, dtype=torch.uint8, device=cx.device) for _ in range(n)]

    def one_pass():
        for W, b in zip(Ws, blobs):
            C.cq_encode(W, 2, cb, blob=b)

    with torch.cuda.stream(stream):
        one_pass()
    stream.synchronize()
    g = graph_of(torch, stream, one_pass)
    Ke = 200
    ms = cx.timed(g.replay, Ke) / Ke
    elems = n * out * n_in
    algo = elems * 4 + n * nb
    gbs = algo / (ms * 1e-3) / 1e9
    for i in range(n):
        rows = sample_rows(out, 4) if i else sample_rows(out, 16)
        cx.samples.add(("encode",), "encode", W=Ws[i][torch.from_numpy(rows).to(cx.device)].cpu().numpy(),
                       blob=host_sub_blob(blobs[i].cpu().numpy(), out, n_in, 2, rows), bits=2, group=128, cb=cb)
    del Ws, g
    res = {"metric": f"CQ2 encode GB/s ({n} fp32 8192x8192 with 1% outliers -> codes + fp16 norms)",
           "value": round(cx.world * gbs, 1), "unit": "GB/s", "ms_per_step": round(ms, 3), "steps": Ke,
           "warmup": 2, "launches_per_step": n, "l2": "inputs larger than L2 (4.3 GB of fp32 per step)",
           "roofline": hbm_roofline(gbs, cx.peaks, cx.peak_kind, ncu_traffic("encode_cq2"),
                                    kernel="encode_kernel<2,1>", algorithmic_bytes_per_launch=algo // n)}

    # ---- the container round trip and a GEMV over a reloaded blob ----
    host = [b.cpu().numpy() for b in blobs]
    cb28 = np.concatenate([cb, C.cq_codebook_init(3), C.cq_codebook_init(4)]).astype(np.float32)
    tmpdir = tempfile.mkdtemp(prefix="cq_bench_")
    path = os.path.join(tmpdir, "outliers.cact")
    t0 = time.perf_counter()
    C.cq_cact_write(path, [dict(dtype=3, shape=(out, n_in), data=h.tobytes(), group=128, bits=2) for h in host],
                    cb28, 128)
    t1 = time.perf_counter()
    file_bytes = os.path.getsize(path)
    with C.cq_cact_open(path) as r:
        t2 = time.perf_counter()
        same = len(r) == n and all(r.tensor(i).data == host[i].tobytes() for i in range(n))
        pick = n - 1
        t = r.tensor(pick)
        cb_file = r.codebook()[:4]
    os.remove(path)
    os.rmdir(tmpdir)
    blob_re = torch.frombuffer(bytearray(t.data), dtype=torch.uint8).to(cx.device)
    x = S.normal((1, n_in), 8100 + pick, device=cx.device)
    y = C.cq_gemv(blob_re, out, n_in, 2, cb_file, x)
    torch.cuda.synchronize()
    rows = sample_rows(out, 32)
    cx.samples.add(("encode", "reload"), "gemv", blob=host_sub_blob(np.frombuffer(t.data, dtype=np.uint8), out,
                                                                      n_in, 2, rows),
                   rows=rows, n_in=n_in, bits=2, group=128, cb=cb_file, x=x.cpu().numpy().astype(np.float64),
                   y=y.cpu().numpy()[:, rows])
    res["reload"] = {"file_bytes": file_bytes, "tensors": n, "write_s": round(t1 - t0, 3),
                     "open_s": round(t2 - t1, 3), "bytes_identical": bool(same), "gemv_matrix": pick,
                     "gemv": "batch 1 on the reloaded blob, codebook read from the file",
                     "gemv_kernel": gemv_kernel_name(out, n_in, 2, 1)}
    return res


def bench_gather(cx, n=65536):
    """Row-gather dequantisation: n random token ids into the tied 8192 x 512
    CQ4 embedding/logit table of the Needle-shaped set (fp32 rows out). The
    steps rotate through output buffers whose footprint is >= 4x L2."""
    C, S, torch, stream = cx.C, cx.S, cx.torch, cx.stream
    out, n_in = 8192, 512
    cb = C.cq_codebook_init(4)
    nb = C.cq_packed_bytes(out, n_in, 128, 4)
    blob = torch.from_numpy(S.random_blob(out * n_in * 4 // 8, out * (n_in // 128), 74)).to(cx.device)
    assert blob.numel() == nb
    g_ = torch.Generator(device="cpu").manual_seed(75)
    idx = torch.randint(0, out, (n,), generator=g_, dtype=torch.int32).to(cx.device)
    obytes = n * n_in * 4
    R = copies_for(obytes, cx.l2) + 1
    dsts = [torch.empty((n, n_in), dtype=torch.float32, device=cx.device) for _ in range(R)]
    with torch.cuda.stream(stream):
        for d in dsts:
            C.cq_gather_rows(blob, out, n_in, 4, cb, idx, dst=d)
    stream.synchronize()
    C.cq_device_status(cx.device)

    def steps():
        for d in dsts:
            C.cq_gather_rows(blob, out, n_in, 4, cb, idx, dst=d)

    g = graph_of(torch, stream, steps)
    reps = max(1, 40 // R)
    ms = cx.timed(g.replay, reps) / (reps * R)
    C.cq_device_status(cx.device)
    row_bytes = nb // out
    algo = n * (row_bytes + 4 * n_in + 4)
    gbs = algo / (ms * 1e-3) / 1e9
    import numpy as np
    pick = sample_rows(n, 64)
    rows = idx.cpu().numpy()[pick]
    cx.samples.add(("gather",), "gather", blob=host_sub_blob(blob.cpu().numpy(), out, n_in, 4, rows), n_in=n_in,
                   bits=4, cb=cb, got=dsts[-1].cpu().numpy()[pick], nrows=len(rows))
    del dsts, g
    return {"metric": f"CQ4 row gather GB/s ({n} token ids into the 8192x512 embedding table -> fp32 rows)",
            "value": round(cx.world * gbs, 1), "unit": "GB/s", "ms_per_step": round(ms, 4), "steps": reps * R,
            "warmup": 1, "l2": f"{R} rotating output buffers ({R * obytes / 1e6:.0f} MB >= 4x L2)",
            "roofline": hbm_roofline(gbs, cx.peaks, cx.peak_kind, ncu_traffic("gather_cq4"),
                                     kernel="gather_rows_kernel<4,128>", algorithmic_bytes_per_launch=algo)}


def bench_kv(cx):
    """Decode-step attention over CQ KV caches: 256 sequences x 8192 cached
    tokens in the Needle 3 attention geometry, CQ2 keys and values, one call
    per step. Four copies of the caches (different seeds) rotate, so a
    step's 144 MB never sit in L2 from the steps before."""
    import numpy as np
    C, S, torch, stream = cx.C, cx.S, cx.torch, cx.stream
    g = S.KV_GEOM
    Hq, Hkv, dk, dv = g["n_q_heads"], g["n_kv_heads"], g["head_dim_k"], g["head_dim_v"]
    T, nseq, bits = S.KV_TOKENS, S.KV_SEQS, S.KV_BITS
    cb = C.cq_codebook_init(bits)
    scale = 1.0 / math.sqrt(dk)
    sets = []
    nsets = 4
    for r in range(nsets):
        items = []
        for i in range(nseq):
            kc = torch.from_numpy(S.kv_cache_blob(T, Hkv * dk, bits, 20000 * r + 5000 + i)).to(cx.device)
            vc = torch.from_numpy(S.kv_cache_blob(T, Hkv * dv, bits, 20000 * r + 6000 + i)).to(cx.device)
            q = S.normal((Hq, dk), 20000 * r + 7000 + i).to(cx.device)
            items.append(dict(k_cache=kc, v_cache=vc, cap=T, n_tokens=T, q=q,
                              o=torch.empty((Hq, dv), dtype=torch.float32, device=cx.device)))
        sets.append(items)
    with torch.cuda.stream(stream):  # grows the workspace before capture
        for items in sets:
            C.cq_kv_attend(items, Hq, Hkv, dk, dv, bits, bits, cb, cb, scale)
    stream.synchronize()

    def steps():
        for items in sets:
            C.cq_kv_attend(items, Hq, Hkv, dk, dv, bits, bits, cb, cb, scale)

    gr = graph_of(torch, stream, steps)
    reps = 10
    ms = cx.timed(gr.replay, reps) / (nsets * reps)
    kb = C.cq_packed_bytes(T, Hkv * dk, 128, bits)
    vb = C.cq_packed_bytes(T, Hkv * dv, 128, bits)
    algo = nseq * (kb + vb + 4 * Hq * dk + 4 * Hq * dv)
    gbs = algo / (ms * 1e-3) / 1e9
    tok = nseq * T / (ms * 1e-3)
    for i in (0, nseq - 1):
        it = sets[-1][i]
        cx.samples.add(("kv",), "kv", k=it["k_cache"].cpu().numpy(), v=it["v_cache"].cpu().numpy(), T=T,
                       q=it["q"].cpu().numpy(), o=it["o"].cpu().numpy(), geom=(Hq, Hkv, dk, dv), bits=bits, cb=cb,
                       scale=scale)
    return {"metric": f"CQ{bits} KV-cache decode attention GB/s ({nseq} sequences x {T} tokens, "
                      f"{Hq} query heads of {dk} over {Hkv} KV heads, values of {dv})",
            "value": round(cx.world * gbs, 1), "unit": "GB/s", "ms_per_step": round(ms, 4),
            "cached_tokens_per_s": round(cx.world * tok, 1), "steps": nsets * reps, "warmup": nsets,
            "l2": f"{nsets} cache copies rotate ({nsets * algo / 1e6:.0f} MB cycle)",
            "roofline": hbm_roofline(gbs, cx.peaks, cx.peak_kind, ncu_traffic("kv_attend"),
                                     kernel="kv_attend_warp_kernel<3>", algorithmic_bytes_per_launch=algo)}


def bench_g64_gemm(cx, M=2048):
    """The GEMM at M=2048 int8 tokens over group-64 CQ2 and binary weights
    beside group-128 CQ2: 16 matrices of 4096 x 512 (weights rotated back on
    chip) and 4 of 4096 x 4096 (rotated activations), one grouped call per
    step; the fp32 outputs (512 MB and 128 MB) exceed L2."""
    import numpy as np
    C, S, torch, stream = cx.C, cx.S, cx.torch, cx.stream
    res = {}
    cases = (("gemm_cq2_group64_in512", 64, 2, 16, 512), ("gemm_binary_in512", 128, 1, 16, 512),
             ("gemm_cq2_group128_in512", 128, 2, 16, 512), ("gemm_binary_in4096", 128, 1, 4, 4096),
             ("gemm_cq2_group128_in4096", 128, 2, 4, 4096))
    for name, group, bits, nmat, n_in in cases:
        out = 4096
        cb = C.cq_codebook_init(bits, group)
        nb = C.cq_packed_bytes(out, n_in, group, bits)
        Xq, xs = C.cq_act_quant_int8(S.normal((M, n_in), 33000 + n_in, device=cx.device))
        items = []
        for i in range(nmat):
            blob = torch.from_numpy(S.random_blob(out * n_in * bits // 8, out * n_in // group,
                                                  34000 + 100 * bits + group + i)).to(cx.device)
            items.append(dict(blob=blob, out=out, **{"in": n_in}, bits=bits, codebook=cb, Xq=Xq, x_scale=xs,
                              group=group, Y=torch.empty((M, out), dtype=torch.float32, device=cx.device)))
        with torch.cuda.stream(stream):
            for _ in range(3):
                C.cq_gemm_grouped(items)
        stream.synchronize()

        def steps():
            for _ in range(5):
                C.cq_gemm_grouped(items)

        g = graph_of(torch, stream, steps)
        reps = 20
        ms = cx.timed(g.replay, reps) / (5 * reps)
        C.cq_device_status(cx.device)
        flops = 2.0 * M * out * n_in * nmat
        tflops = flops / (ms * 1e-3) / 1e12
        toks, rows = sample_rows(M, 4), sample_rows(out, 8)
        td, rd = torch.from_numpy(toks).to(cx.device), torch.from_numpy(rows).to(cx.device)
        x = Xq[td].cpu().numpy().astype(np.float64) * xs[td].cpu().numpy().astype(np.float64)[:, None]
        per = [dict(blob=host_sub_blob(it["blob"].cpu().numpy(), out, n_in, bits, rows, group), rows=rows,
                    n_in=n_in, bits=bits, group=group, cb=np.asarray(cb), x=x,
                    y=it["Y"][td][:, rd].cpu().numpy()) for it in items[:2]]
        cx.samples.add(("group64_binary", name), "gemm", per=per)
        res[name] = {"metric": f"CQ GEMM TFLOP/s at M={M}, {nmat} x {out}x{n_in}, group {group}, {bits}-bit codes",
                     "value": round(cx.world * tflops, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 5),
                     "steps": 5 * reps, "packed_bytes_per_step": nmat * nb,
                     "l2": f"outputs larger than L2 (fp32 Y, {4 * M * out * nmat / 1e6:.0f} MB per step)",
                     "tensor_view": {"achieved": round(tflops, 2), "peak": cx.peaks["bf16_tflops"], "unit": "TFLOP/s",
                                     "frac": round(tflops / cx.peaks["bf16_tflops"], 4),
                                     "peak_source": cx.peak_kind + " (bf16 dense; fp16 operands run at the same rate)"}}
        del items, g
    return res


def bench_g64(cx):
    """Group-64 CQ2 and binary (group 128) weights: one grouped GEMV launch
    over 64 matrices of 4096 x 4096 (batch 1, fp32 activations), the set
    larger than L2, plus the encoder on 8 x 8192^2 at group 64 CQ2."""
    C, S, torch, stream = cx.C, cx.S, cx.torch, cx.stream
    res = {}
    for name, group, bits in (("cq2_group64", 64, 2), ("binary_group128", 128, 1), ("cq2_group128", 128, 2)):
        out = n_in = 4096
        cb = C.cq_codebook_init(bits, group)
        nb = C.cq_packed_bytes(out, n_in, group, bits)
        ip = (n_in + group - 1) // group * group
        items = []
        for i in range(64):
            blob = torch.from_numpy(S.random_blob(out * ip * (2 if bits == 5 else bits) // 8, out * ip // group,
                                                  30000 + 100 * bits + i)).to(cx.device)
            x = S.normal((1, n_in), 31000 + i).to(cx.device)
            items.append(dict(blob=blob, out=out, **{"in": n_in}, bits=bits, codebook=cb, x=x, group=group,
                              y=torch.empty((1, out), dtype=torch.float32, device=cx.device)))
        plan = C.GemvPlan(items)
        with torch.cuda.stream(stream):
            for _ in range(3):
                plan.run(stream)
        stream.synchronize()

        def steps():
            for _ in range(10):
                plan.run(stream)

        g = graph_of(torch, stream, steps)
        reps = 10
        ms = cx.timed(g.replay, reps) / (10 * reps)
        algo = 64 * (nb + 4 * n_in + 4 * out)
        gbs = algo / (ms * 1e-3) / 1e9
        import numpy as np
        rows = sample_rows(out, 16)
        cx.samples.add(("group64_binary", name), "gemv",
                       blob=host_sub_blob(items[0]["blob"].cpu().numpy(), out, n_in, bits, rows, group), rows=rows,
                       n_in=n_in, bits=bits, group=group, cb=np.asarray(cb),
                       x=items[0]["x"].cpu().numpy().astype(np.float64), y=items[0]["y"].cpu().numpy()[:, rows])
        res[name] = {"metric": f"GEMV GB/s, 64 x 4096x4096, group {group}, {bits}-bit codes, batch 1",
                     "value": round(cx.world * gbs, 1), "unit": "GB/s", "ms_per_step": round(ms, 4),
                     "steps": 10 * reps, "packed_bytes_per_step": 64 * nb,
                     "l2": f"one set of 64 matrices ({64 * nb / 1e6:.0f} MB > L2)",
                     "roofline": hbm_roofline(gbs, cx.peaks, cx.peak_kind,
                                              ncu_traffic("gemv_split") if name == "cq2_group128" else
                                              ncu_traffic("gemv_split_g64") if name == "cq2_group64" else None,
                                              kernel=gemv_kernel_name(out, n_in, bits, 1, group),
                                              algorithmic_bytes_per_launch=algo)}
        del items, plan, g
    res.update(bench_g64_gemm(cx))
    # encoder at group 64
    cb = C.cq_codebook_init(2, 64)
    ne = 8
    Ws = [S.normal((8192, 8192), 32000 + i, S.W_STD, device=cx.device) for i in range(ne)]
    blobs = [torch.empty(C.cq_packed_bytes(8192, 8192, 64, 2), dtype=torch.uint8, device=cx.device)
             for _ in range(ne)]

    def one_pass():
        for W, bl in zip(Ws, blobs):
            C.cq_encode(W, 2, cb, group=64, blob=bl)

    with torch.cuda.stream(stream):
        one_pass()
    stream.synchronize()
    g = graph_of(torch, stream, one_pass)
    reps = 400
    ms = cx.timed(g.replay, reps) / (reps * ne)
    algo = 8192 * 8192 * 4 + blobs[0].numel()
    gbs = algo / (ms * 1e-3) / 1e9
    rows = sample_rows(8192, 4)
    cx.samples.add(("group64_binary", "encode_cq2_group64"), "encode",
                   W=Ws[0][torch.from_numpy(rows).to(cx.device)].cpu().numpy(),
                   blob=host_sub_blob(blobs[0].cpu().numpy(), 8192, 8192, 2, rows, 64), bits=2, group=64, cb=cb)
    res["encode_cq2_group64"] = {"metric": "encode GB/s, 8192x8192 fp32 -> CQ2 at group 64",
                                 "value": round(cx.world * gbs, 1), "unit": "GB/s", "ms_per_matrix": round(ms, 4),
                                 "launches": reps * ne, "l2": f"{ne} input matrices rotate (2.1 GB)",
                                 "roofline": hbm_roofline(gbs, cx.peaks, cx.peak_kind, None,
                                                          kernel="encode_g64_kernel<2,1>",
                                                          algorithmic_bytes_per_launch=algo)}
    return res


# ------------------------------------------------------------ CPU oracle
# The one leg of this script that runs the oracle (test infrastructure):
# after every GPU part is done, on rank 0 at N=1. It times the oracle as the
# CPU baseline and recomputes the outputs the GPU parts sampled.

def host_cpu():
    """(logical cores usable by this process, CPU model string)."""
    try:
        cores = len(os.sched_getaffinity(0))
    except Exception:
        cores = os.cpu_count() or 1
    model = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
        if not model:
            for line in out.splitlines():
                if line.lower().startswith(("vendor id", "architecture")):
                    model += line.split(":", 1)[1].strip() + " "
    except Exception:
        pass
    import platform
    return cores, (model.strip() or platform.processor() or platform.machine())


def oracle_units(mats, blobs, cbs, xts, max_rows=512):
    """The oracle's product over a matrix set, cut into units of at most
    max_rows output rows: (matrix index, first row, sub-blob, rows, in, bits,
    codebook, activation as fp64 [B, in])."""
    import numpy as np
    units = []
    for i, (m, blob) in enumerate(zip(mats, blobs)):
        for r0 in range(0, m.out, max_rows):
            rows = np.arange(r0, min(m.out, r0 + max_rows))
            units.append((i, r0, host_sub_blob(blob, m.out, m.n_in, m.bits, rows), len(rows), m.n_in, m.bits,
                          cbs[m.bits], xts[i]))
    return units


def run_unit(u):
    """One unit of oracle work: dequantise (explicit Hadamard, fp64), then
    the dense fp64 product. Returns (matrix, first row, y, bound, bytes)."""
    import oracle as O
    i, r0, sub, nrows, n_in, bits, cb, xt = u
    What = O.dequant(sub, nrows, n_in, bits, cb)
    y, bd = O.matmul(What, xt)
    return i, r0, y, bd, sub.size


def time_units(units, threads, budget_s=None):
    """Runs units in order (one thread) or over a pool of `threads` (the C
    oracle releases the GIL), stopping once budget_s is spent (single
    thread) -- returns (results, bytes, seconds)."""
    from concurrent.futures import ThreadPoolExecutor
    t0 = time.perf_counter()
    res, nbytes = [], 0
    if threads <= 1:
        for u in units:
            r = run_unit(u)
            res.append(r)
            nbytes += r[4]
            if budget_s is not None and time.perf_counter() - t0 >= budget_s:
                break
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            for r in ex.map(run_unit, units):
                res.append(r)
                nbytes += r[4]
    return res, nbytes, time.perf_counter() - t0


def _product_stats(y, y_ref, bound):
    """max |y - y_ref| / bound, min cosine over the rows of y (the batch
    rows), and whether the product tolerance holds."""
    import numpy as np
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.atleast_2d(y_ref)
    bound = np.atleast_2d(bound)
    y = y.reshape(y_ref.shape)
    err = np.abs(y - y_ref)
    worst = float((err / np.maximum(bound, 1e-300)).max()) if err.size else 0.0
    cmin = 1.0
    for b in range(y.shape[0]):
        ny, nr = np.linalg.norm(y[b]), np.linalg.norm(y_ref[b])
        if nr > 0:
            cmin = min(cmin, float(np.dot(y[b], y_ref[b]) / (ny * nr)))
    ok = bool(np.all(err <= 2e-3 * bound + 1e-30)) and cmin >= 0.99999
    return worst, cmin, ok


def _merge_products(stats):
    worst = max((s[0] for s in stats), default=0.0)
    cmin = min((s[1] for s in stats), default=1.0)
    return {"max_err_over_bound": float(f"{worst:.4g}"), "min_cosine": round(cmin, 9),
            "tolerance": "|y - y_ref| <= 2e-3 * sum|w||x| per element, cosine >= 0.99999",
            "pass": all(s[2] for s in stats)}


def _encode_stats(W, blob, bits, group, cb):
    """Encoder parity of sampled rows: codes bit-exact away from decision
    boundaries (coordinates within 1e-6 of one are counted), fp16 norms
    bit-exact."""
    import numpy as np

    import oracle as O
    ref, flags, _ = O.encode(W, bits, cb, group)
    out, n_in = W.shape
    cg, ng = O.unpack(blob, out, n_in, bits, group)
    cr, nr = O.unpack(ref, out, n_in, bits, group)
    diff = cg != cr
    return dict(coords=int(cg.size), boundary=int(flags.sum()), boundary_mismatch=int((diff & (flags != 0)).sum()),
                code_mismatch=int((diff & (flags == 0)).sum()), norms=int(ng.size), norm_mismatch=int((ng != nr).sum()))


def _merge_encode(stats):
    tot = {k: sum(s[k] for s in stats) for k in stats[0]}
    tot["pass"] = tot["code_mismatch"] == 0 and tot["norm_mismatch"] == 0
    tot["rule"] = "codes bit-exact except within 1e-6 of a decision boundary (counted); fp16 norms bit-exact"
    return tot


def _put(result, path, key, value):
    node = result
    for p in path:
        node = node.setdefault(p, {})
    node[key] = value


def oracle_leg(result, samples, budget_s=10.0):
    import numpy as np

    import oracle as O
    sys.path.insert(0, ROOT)
    from tests.gpu_helpers import attention_bound, gather_bound

    cores, model = host_cpu()
    t_leg = time.perf_counter()
    # ---- 1. CPU baseline on the decode step's own blobs and activations ----
    dec = next(s for s in samples.items if s["kind"] == "decode")["wl"]
    mats = dec["mats"]
    xts = [(dec["Xq"][m.act:m.act + 1].astype(np.float64) * np.float64(dec["xs"][m.act])) for m in mats]
    units = oracle_units(mats, dec["blobs"], dec["cbs"], xts)
    res1, b1, t1 = time_units(units, 1, budget_s)
    resn, bn, tn = time_units(units, cores)
    reps = 1
    while tn < 2.0 and reps < 64:  # repeat the all-cores pass to a measurable time
        _, b2, t2 = time_units(units, cores)
        bn, tn, reps = bn + b2, tn + t2, reps + 1
    packed = sum(b.size for b in dec["blobs"])
    result["cpu_baseline"] = {
        "value": round(bn / tn / 1e9, 6), "unit": "GB/s", "cores": cores, "kind": "oracle",
        "cpu_model": model,
        "sample": f"oracle dequantise (explicit 128x128 Hadamard, fp64) + fp64 matmul over the whole decode step "
                  f"({packed} packed bytes, {len(units)} row blocks as threads' work items), {reps} pass(es) in "
                  f"{tn:.2f} s on {cores} threads",
        "single_thread": {"value": round(b1 / t1 / 1e9, 6), "unit": "GB/s", "cores": 1,
                          "sample": f"{b1} packed bytes of the same step in {t1:.2f} s"}}
    # ---- 2. parity of the decode step: every output against the oracle ----
    yref = [np.zeros(m.out) for m in mats]
    bref = [np.zeros(m.out) for m in mats]
    for i, r0, y, bd, _ in resn:
        yref[i][r0:r0 + y.shape[1]] = y[0]
        bref[i][r0:r0 + y.shape[1]] = bd[0]
    par = _merge_products([_product_stats(dec["y"][i], yref[i], bref[i]) for i in range(len(mats))])
    par["outputs_checked"] = int(sum(m.out for m in mats))
    par["encode"] = _merge_encode([_encode_stats(W, host_sub_blob(dec["blobs"][i], m.out, m.n_in, m.bits, rows),
                                                 m.bits, 128, dec["cbs"][m.bits])
                                   for i, (m, (rows, W)) in enumerate(zip(mats, dec["w_rows"]))])
    result["parity"] = par
    # ---- 3. parity of every other sampled workload ----
    groups = {}
    for s in samples.items:
        if s["kind"] == "decode":
            continue
        groups.setdefault((s["path"], s["kind"]), []).append(s)
    for (path, kind), ss in groups.items():
        if kind == "encode":
            st = _merge_encode([_encode_stats(s["W"], s["blob"], s["bits"], s["group"], s["cb"]) for s in ss])
            _put(result, path, "parity", st)
        elif kind == "gemv":
            stats = []
            for s in ss:
                What = O.dequant(s["blob"], len(s["rows"]), s["n_in"], s["bits"], s["cb"], s["group"])
                y_ref, bd = O.matmul(What, s["x"])
                stats.append(_product_stats(s["y"], y_ref, bd))
            st = _merge_products(stats)
            st["outputs_checked"] = int(sum(s["y"].size for s in ss))
            _put(result, path, "parity", st)
        elif kind == "gemm":
            stats, n = [], 0
            for s in ss:
                for p in s["per"]:
                    What = O.dequant(p["blob"], len(p["rows"]), p["n_in"], p["bits"], p["cb"], p.get("group", 128))
                    y_ref, bd = O.matmul(What, p["x"])
                    stats.append(_product_stats(p["y"], y_ref, bd))
                    n += p["y"].size
            st = _merge_products(stats)
            st["outputs_checked"] = n
            _put(result, path, "parity", st)
        elif kind == "gather":
            worst = 0.0
            for s in ss:
                ref = O.dequant(s["blob"], s["nrows"], s["n_in"], s["bits"], s["cb"])
                bd = gather_bound(s["blob"], s["nrows"], s["n_in"], s["bits"], s["cb"], np.arange(s["nrows"]))
                worst = max(worst, float((np.abs(s["got"].astype(np.float64) - ref) / bd).max()))
            _put(result, path, "parity", {"rows_checked": int(sum(s["nrows"] for s in ss)),
                                          "max_err_over_bound": float(f"{worst:.4g}"), "pass": worst <= 1.0,
                                          "tolerance": "|err| <= 1e-6 * n/sqrt(128) * sum_k |c[q_k]| per group"})
        elif kind == "kv":
            worst, cmin = 0.0, 1.0
            for s in ss:
                Hq, Hkv, dk, dv = s["geom"]
                o_ref, P, Kh, Vh = O.kv_attend(s["k"], s["v"], s["T"], s["T"], s["q"].astype(np.float64), Hkv, dk, dv,
                                               s["bits"], s["bits"], s["cb"], s["cb"], np.float32(s["scale"]))
                bd = attention_bound(Kh, Vh, s["q"].astype(np.float64), P, o_ref, Hkv, s["scale"])
                o = s["o"].astype(np.float64)
                worst = max(worst, float((np.abs(o - o_ref) / np.maximum(bd, 1e-300)).max()))
                for b in range(Hq):
                    cmin = min(cmin, float(np.dot(o[b], o_ref[b]) / (np.linalg.norm(o[b]) * np.linalg.norm(o_ref[b]))))
            _put(result, path, "parity", {"sequences_checked": len(ss), "max_err_over_bound": float(f"{worst:.4g}"),
                                          "min_cosine": round(cmin, 9), "pass": worst <= 1.0 and cmin >= 0.99999,
                                          "tolerance": "product-rule bound on the softmax-weighted value sum, "
                                                       "cosine >= 0.99999 per head"})
    result["cpu_baseline"]["oracle_leg_s"] = round(time.perf_counter() - t_leg, 1)


def reference_units():
    """The decode step's geometry with seeded random blobs and the seeded
    activations (CPU generators): the reference arm's workload."""
    import numpy as np

    import oracle as O
    import synthetic as S
    mats = S.decode_step_mats()
    cbs = {b: O.analytic_codebook(b) for b in (2, 4)}
    blobs, xts = [], []
    acts = {}
    for i, m in enumerate(mats):
        ip = O.in_padded(m.n_in)
        blobs.append(S.random_blob(m.out * ip * O.width(m.bits) // 8, m.out * ip // 128, 9000 + i))
        if m.act not in acts:
            q, s = O.act_quant_int8(S.decode_activation(m.act).numpy())
            acts[m.act] = q.astype(np.float64) * s.astype(np.float64)[:, None]
        xts.append(acts[m.act])
    return oracle_units(mats, blobs, cbs, xts)


def run_reference(args):
    world, rank, _ = rank_context()
    if rank != 0:  # the oracle runs on rank 0 alone; the other ranks exit without work
        return
    cores, model = host_cpu()
    units = reference_units()
    K, Wm = args.steps, args.warmup
    K_run = min(K, 200)
    per_step = max(0.05, min(2.0, 120.0 / max(1, K_run + Wm)))
    # calibrate: units per step so that a step takes about per_step seconds
    _, _, t = time_units(units, cores)
    n_per = max(1, min(len(units), int(len(units) * per_step / max(t, 1e-6))))
    for w in range(min(Wm, 3)):
        time_units(units[:n_per], cores)
    tot_b, tot_t = 0, 0.0
    for k in range(K_run):
        off = (k * n_per) % len(units)
        chunk = (units[off:] + units[:off])[:n_per]
        _, b, t = time_units(chunk, cores)
        tot_b += b
        tot_t += t
    v = tot_b / tot_t / 1e9
    res = {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "GB/s", "n_gpus": world,
           "steps": K_run, "warmup": Wm, "ms_per_step": round(1e3 * tot_t / K_run, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": WORKLOAD, "sample": f"{n_per} of the step's {len(units)} row blocks per step"},
           "cpu_baseline": {"value": round(v, 6), "unit": "GB/s", "cores": cores, "kind": "oracle",
                            "cpu_model": model,
                            "sample": "decode-step row blocks in order, oracle dequantise + fp64 matmul, "
                                      f"threads over row blocks ({cores})"},
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
    ap.add_argument("--only", default="all",
                    choices=["all", "decode", "gemm", "gemm_small", "encode", "gather", "kv", "g64", "sweep",
                             "single"],
                    help="time one part alone and print its JSON object (profiling)")
    ap.add_argument("--cpu-seconds", type=float, default=8.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_cq(args)


if __name__ == "__main__":
    main()
