"""Bench of the quantized-weight matvec path on GB300.

One step = one pass of the whole path over one batch-1 decode-shaped input,
with every input already resident in HBM:

  1. cq_prepare        x[500] -> prepared[512]        (CQ 2-bit vocabulary matrix)
  2. cq_matvec         32768 x 512, 2-bit, group 128  -> logits[32768]
  3. cq_dequantize_row 64 row ids                     -> embeddings[64, 500]
  4. f8_matvec         245760 x 4096 E4M3, E8M0 scales [1920, 32] -> head[245760]

metric: weight GB/s (algorithmic bytes: packed weights + norms / scales +
codebook + activations in + results out) per second, plus microseconds per
matvec and the fraction of HBM bandwidth of the dominant kernel.  Each step
streams ~1.01 GB, more than the 129 MB L2, so every step starts L2-cold for
the weights.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) each rank runs an independent replica on its own GPU
(the matvec has no exchange step); the time is the max over ranks and the
value counts the bytes of all ranks.  --impl reference times the CPU oracle
on the host cores over a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "batch-1 quantized matvec: weight GB/s and % of GB300 HBM peak; µs per matvec"
WORKLOAD = ("decode pair, batch 1: CQ 2-bit vocabulary projection 32768x512 (input 500, "
            "group 128) with prepare and a 64-row gather + F8 E4M3 head 245760x4096 "
            "(E8M0 scales [1920,32])")
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


# --------------------------------------------------------------------------
# algorithmic bytes
# --------------------------------------------------------------------------

# The pages' own CPU figures, quoted with their hardware as context only
# (none is a GPU number, and none measures this metric on this workload).
PAGES_CPU_CONTEXT = [
    {"figure": "0.19 s/token", "what": "structural decode of the MoE path only (no attention, "
     "no head), at the read floor", "hardware": "the 'acer' box (CPU)",
     "source": "ds4f-disk issue #6, milestone summary"},
    {"figure": "0.1-0.2 s/token", "what": "projected ~246k x 4096 F8 head (~2 GFLOP/token), "
     "threaded, resident", "hardware": "the 'acer' box (CPU)",
     "source": "ds4f-disk issue #6, 'Expected cost on the acer'"},
    {"figure": "1.5-2 tok/s (0.5-0.8 s/token)", "what": "projected full single-stream decode",
     "hardware": "the 'acer' box (CPU)", "source": "ds4f-disk issue #6, 'Expected cost on the acer'"},
    {"figure": "0.29 s/token; head ~0.05 s/token", "what": "measured decode after the SIMD "
     "I8/F8 matvecs", "hardware": "the 'acer' box (CPU)", "source": "ds4f-disk issue #6, step 4"},
    {"figure": "4.06 GFLOP/s (scalar 1.32)", "what": "F8 E4M3 + E8M0 matvec, NEON, "
     "'decode-bound'", "hardware": "Apple M4 (CPU)", "source": "ds4f-disk issue #6, step 4"},
    {"figure": "27.1 GFLOP/s (scalar 1.94)", "what": "I8 matvec with per-16 E8M0 scales, NEON",
     "hardware": "Apple M4 (CPU)", "source": "ds4f-disk issue #6, step 4"},
]


def cq_matvec_bytes(out, P, G, bits, batch=1):
    rb = (P * bits + 7) // 8
    return out * rb + out * (P // G) * 2 + (1 << bits) * 4 + batch * P * 4 + batch * out * 4


def cq_prepare_bytes(inp, P, batch=1):
    return batch * (inp + P) * 4


def cq_gather_bytes(n, inp, P, G, bits):
    rb = (P * bits + 7) // 8
    return n * 4 + n * (rb + (P // G) * 2) + (1 << bits) * 4 + n * inp * 4


def f8_bytes(R, C, SR, SC, batch=1):
    return R * C + SR * SC + batch * C * 4 + batch * R * 4


def step_bytes(cq, f8):
    return {
        "cq_prepare": cq_prepare_bytes(cq.input, cq.input_padded),
        "cq_matvec": cq_matvec_bytes(cq.output, cq.input_padded, cq.group, cq.bits),
        "cq_dequantize_row": cq_gather_bytes(len(cq.rows), cq.input, cq.input_padded, cq.group,
                                             cq.bits),
        "f8_matvec": f8_bytes(f8.R, f8.C, f8.SR, f8.SC),
    }


def make_inputs():
    from quantized_weight_matvec_gb300 import synth
    cq = synth.workload_inputs("cq2_vocab")
    f8 = synth.workload_inputs("f8_head", batch=1)
    return cq, f8


# --------------------------------------------------------------------------
# distributed helpers (replicas)
# --------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def barrier(d):
    if d is not None:
        d.barrier()


def max_over_ranks(value: float, d) -> float:
    """Max of a float over all ranks (identity on one rank)."""
    if d is None:
        return value
    import torch
    dev = "cuda" if d.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    d.all_reduce(t, op=d.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------
# clocks
# --------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
             "utilization.gpu")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="qmv_clocks_", suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), max=float(parts[2]), power=float(parts[3]),
                                 active=parts[4], hw=parts[5], hwt=parts[6], swt=parts[7],
                                 pcap=parts[8], util=float(parts[9])))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        load = [r for r in rows if r["util"] >= 50] or rows
        reasons = set()
        for r in load:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in load),
                "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(load),
                "power_w_max": max(r["power"] for r in rows)}


# --------------------------------------------------------------------------
# roofline inputs
# --------------------------------------------------------------------------

def measured_hbm_gbs():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# What the batch-1 head kernel (f8_fast_kernel) is compiled from.
TRAFFIC_SOURCES = ("f8_kernels.cu", "f8_common.cuh", "device_common.cuh", "qmv_internal.h")


def kernel_source_hash():
    h = hashlib.sha256()
    for name in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, "quantized_weight_matvec_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def ncu_traffic():
    """DRAM bytes per f8_matvec launch from the committed ncu summary, or None
    if the kernel source changed since it was captured."""
    path = os.path.join(ROOT, "profiles", "f8_head_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    if rec.get("source_sha256") != kernel_source_hash():
        return None
    return rec.get("dram_bytes_per_launch")


# --------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------

def cq_matvec_alone_us(torch, qmv, cq, dev, prepared, logits):
    """Median microseconds per cq_matvec call (the CQ 2-bit vocabulary
    projection), L2-cold: a CUDA graph of back-to-back calls, each over its
    own copy of the packed rows and norms (copies totalling > 2x L2)."""
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    per = cq.packed.nbytes + cq.norms.nbytes
    k = max(2, -(-2 * l2 // per))
    packed = torch.from_numpy(cq.packed).to(dev).unsqueeze(0).repeat(k, 1, 1)
    norms = torch.from_numpy(cq.norms.view(np.int16)).to(dev).unsqueeze(0).repeat(k, 1, 1)
    cb = torch.from_numpy(cq.codebook).to(dev)
    mats = [qmv.CQMatrix(cq.output, cq.input, cq.input_padded, cq.group, cq.bits, packed[i],
                         norms[i], cb) for i in range(k)]
    calls = [(lambda m: lambda sh: qmv.cq_matvec(m.struct, prepared.data_ptr(), 1,
                                                  logits.data_ptr(), sh))(m) for m in mats]
    med, _ = _graph_time(torch, calls)
    del packed, norms, mats
    return med, k


def run_ours(args):
    import torch
    from quantized_weight_matvec_gb300 import qmv

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    d = init_dist(world, "nccl")
    qmv.load()
    cq, f8 = make_inputs()
    nbytes = step_bytes(cq, f8)
    total_bytes = sum(nbytes.values())

    dev = torch.device("cuda", local)
    m = qmv.CQMatrix.from_numpy(cq, device=dev)
    x3 = torch.from_numpy(cq.x).to(dev)
    ids = torch.from_numpy(cq.rows).to(dev)
    w5 = torch.from_numpy(f8.w).to(dev)
    s5 = torch.from_numpy(f8.scale).to(dev)
    x5 = torch.from_numpy(f8.x).to(dev)
    prepared = torch.empty((1, cq.input_padded), dtype=torch.float32, device=dev)
    logits = torch.empty((1, cq.output), dtype=torch.float32, device=dev)
    emb = torch.empty((len(cq.rows), cq.input), dtype=torch.float32, device=dev)
    head = torch.empty((1, f8.R), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    # The CQ chain (prepare -> matvec, and the gather) shares no data with the
    # F8 head: in the timed steps it runs on a second stream beside the head,
    # forked from and joined to the main stream around the timed region.
    side = torch.cuda.Stream(dev)
    names = ["cq_prepare", "cq_matvec", "cq_dequantize_row", "f8_matvec"]

    def check(st, name):
        if st != 0:
            raise RuntimeError("%s failed: %s" % (name, qmv.status_string(st)))

    def step(ev=None, cq_stream=None):
        cs = sh if cq_stream is None else cq_stream.cuda_stream
        if ev is not None:
            ev[0].record(stream)
        check(qmv.cq_prepare(m.struct, x3.data_ptr(), 1, prepared.data_ptr(), cs), names[0])
        if ev is not None:
            ev[1].record(stream)
        check(qmv.cq_matvec(m.struct, prepared.data_ptr(), 1, logits.data_ptr(), cs), names[1])
        if ev is not None:
            ev[2].record(stream)
        check(qmv.cq_dequantize_row(m.struct, ids.data_ptr(), ids.numel(), emb.data_ptr(), 0, cs),
              names[2])
        if ev is not None:
            ev[3].record(stream)
        check(qmv.f8_matvec(w5.data_ptr(), f8.R, f8.C, s5.data_ptr(), f8.SR, f8.SC, x5.data_ptr(),
                            1, head.data_ptr(), sh), names[3])
        if ev is not None:
            ev[4].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # pinned host buffers of the end-to-end pass: activations and row ids
    # in, the three results out (weights stay resident)
    hx3 = torch.from_numpy(cq.x).pin_memory()
    hids = torch.from_numpy(cq.rows).pin_memory()
    hx5 = torch.from_numpy(f8.x).pin_memory()
    hlog = torch.empty(logits.shape, dtype=torch.float32).pin_memory()
    hemb = torch.empty(emb.shape, dtype=torch.float32).pin_memory()
    hhead = torch.empty(head.shape, dtype=torch.float32).pin_memory()

    # Steps are pipelined: device inputs and outputs are double-buffered, the
    # CQ chain runs on a second stream beside the F8 head, host->device copies
    # run on their own stream ahead of the step that reads them, and
    # device->host copies on another, overlapping the next step's kernels.
    # Events keep every buffer's reuse in order.  The device-only timed region
    # runs the same steps without the copies.
    class _Bufs:
        pass

    bufs = []
    for _ in range(2):
        b = _Bufs()
        b.x3, b.ids, b.x5 = torch.empty_like(x3), torch.empty_like(ids), torch.empty_like(x5)
        b.prepared, b.logits = torch.empty_like(prepared), torch.empty_like(logits)
        b.emb, b.head = torch.empty_like(emb), torch.empty_like(head)
        b.ev_in, b.ev_head, b.ev_cq, b.ev_out = (torch.cuda.Event() for _ in range(4))
        bufs.append(b)
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_step(i, copies=True):
        b = bufs[i % 2]
        with torch.cuda.stream(h2d_s):  # after the kernels that last read this buffer
            h2d_s.wait_event(b.ev_head)
            h2d_s.wait_event(b.ev_cq)
            if copies:
                b.x3.copy_(hx3, non_blocking=True)
                b.ids.copy_(hids, non_blocking=True)
                b.x5.copy_(hx5, non_blocking=True)
            b.ev_in.record(h2d_s)
        for st in (side, stream):  # inputs landed; outputs of this buffer read back
            st.wait_event(b.ev_in)
            st.wait_event(b.ev_out)
        ss = side.cuda_stream
        check(qmv.cq_prepare(m.struct, b.x3.data_ptr(), 1, b.prepared.data_ptr(), ss), names[0])
        check(qmv.cq_matvec(m.struct, b.prepared.data_ptr(), 1, b.logits.data_ptr(), ss), names[1])
        check(qmv.cq_dequantize_row(m.struct, b.ids.data_ptr(), b.ids.numel(), b.emb.data_ptr(), 0, ss),
              names[2])
        b.ev_cq.record(side)
        check(qmv.f8_matvec(w5.data_ptr(), f8.R, f8.C, s5.data_ptr(), f8.SR, f8.SC, b.x5.data_ptr(), 1,
                            b.head.data_ptr(), sh), names[3])
        b.ev_head.record(stream)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(b.ev_head)
            d2h_s.wait_event(b.ev_cq)
            if copies:
                hlog.copy_(b.logits, non_blocking=True)
                hemb.copy_(b.emb, non_blocking=True)
                hhead.copy_(b.head, non_blocking=True)
            b.ev_out.record(d2h_s)

    def fork(ev):
        for st in (side, h2d_s, d2h_s):
            st.wait_event(ev)

    def join():
        for st in (side, h2d_s, d2h_s):
            stream.wait_stream(st)

    # timed region: K whole steps in the pipelined form above, without the
    # host copies (inputs resident)
    clocks = ClockSampler(local)
    clocks.start()
    barrier(d)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    for bb in bufs:  # resident inputs in both buffer sets
        bb.x3.copy_(x3)
        bb.ids.copy_(ids)
        bb.x5.copy_(x5)
    warm = torch.cuda.Event()
    warm.record(stream)
    fork(warm)
    for k in range(args.warmup):
        e2e_step(k, copies=False)
    join()
    torch.cuda.synchronize()
    t0.record(stream)
    fork(t0)
    for k in range(args.steps):
        e2e_step(k, copies=False)
    join()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(d)
    clock_info = clocks.stop()
    elapsed_ms = t0.elapsed_time(t1)

    # breakdown pass: up to 200 more steps with an event pair around every call,
    # recorded on the launching stream; each interval includes that call's
    # launch latency, so per-kernel rates here are conservative
    nb = min(args.steps, 200)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(nb)]
    barrier(d)
    torch.cuda.synchronize()
    for k in range(nb):
        step(evs[k])
    torch.cuda.synchronize()
    barrier(d)
    per_kernel_ms = {n: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in evs)
                     for i, n in enumerate(names)}

    # the roofline kernel alone: back-to-back f8_matvec launches between one
    # event pair on its stream (each reads the 1 GB head from HBM: L2-cold)
    nh = min(args.steps, 50)
    h0 = torch.cuda.Event(enable_timing=True)
    h1 = torch.cuda.Event(enable_timing=True)
    barrier(d)
    torch.cuda.synchronize()
    h0.record(stream)
    for _ in range(nh):
        check(qmv.f8_matvec(w5.data_ptr(), f8.R, f8.C, s5.data_ptr(), f8.SR, f8.SC, x5.data_ptr(), 1,
                            head.data_ptr(), sh), names[3])
    h1.record(stream)
    torch.cuda.synchronize()
    barrier(d)
    f8_alone_ms = h0.elapsed_time(h1) / nh

    # the same head at batch 8 (the tcgen05 kernel: raw E4M3 weights by TMA as
    # the MMA's wide operand), seeded activations, back-to-back launches
    x8 = torch.from_numpy(np.random.default_rng(55).standard_normal((8, f8.C)).astype(np.float32)).to(dev)
    head8 = torch.empty((8, f8.R), dtype=torch.float32, device=dev)
    n8 = min(args.steps, 20)
    for _ in range(3):
        check(qmv.f8_matvec(w5.data_ptr(), f8.R, f8.C, s5.data_ptr(), f8.SR, f8.SC, x8.data_ptr(), 8,
                            head8.data_ptr(), sh), names[3])
    torch.cuda.synchronize()
    h0.record(stream)
    for _ in range(n8):
        check(qmv.f8_matvec(w5.data_ptr(), f8.R, f8.C, s5.data_ptr(), f8.SR, f8.SC, x8.data_ptr(), 8,
                            head8.data_ptr(), sh), names[3])
    h1.record(stream)
    torch.cuda.synchronize()
    barrier(d)
    f8_b8_ms = h0.elapsed_time(h1) / n8
    assert torch.isfinite(head8).all()
    del head8, x8

    # the CQ vocabulary projection alone: back-to-back cq_matvec calls over
    # distinct copies of the matrix totalling more than twice the L2 (each
    # call L2-cold), captured in a CUDA graph and replayed, since at ~us per
    # call the host's launch rate would otherwise be what is measured
    cq_alone_us, cq_copies = cq_matvec_alone_us(torch, qmv, cq, dev, prepared, logits)

    # end to end through the C-ABI: the same steps with every step's inputs
    # copied from pinned host memory and its three results copied back
    fork_ev = torch.cuda.Event()
    fork_ev.record(stream)
    fork(fork_ev)
    for k in range(max(3, args.warmup)):
        e2e_step(k)
    join()
    torch.cuda.synchronize()
    barrier(d)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    fork(e0)
    for k in range(args.steps):
        e2e_step(k)
    join()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(d)
    e2e_ms = e0.elapsed_time(e1)
    h2d = hx3.numel() * 4 + hids.numel() * 4 + hx5.numel() * 4
    d2h = (hlog.numel() + hemb.numel() + hhead.numel()) * 4

    # correctness spot check of this run's outputs (cheap, outside timing)
    assert torch.isfinite(head).all() and torch.isfinite(logits).all()

    elapsed_s = max_over_ranks(elapsed_ms / 1e3, d)
    e2e_s = max_over_ranks(e2e_ms / 1e3, d)
    f8_s = max_over_ranks(f8_alone_ms / 1e3, d)
    f8_b8_s = max_over_ranks(f8_b8_ms / 1e3, d)
    cq_s = max_over_ranks(cq_alone_us / 1e6, d)
    cpu = cpu_baseline(cq, f8) if (rank == 0 and world == 1) else None
    if rank != 0:
        if d is not None:
            d.destroy_process_group()
        return
    peak, peak_kind = measured_hbm_gbs()
    f8_achieved = nbytes["f8_matvec"] / f8_s / 1e9
    b8_bytes = f8_bytes(f8.R, f8.C, f8.SR, f8.SC, 8)
    b8_achieved = b8_bytes / f8_b8_s / 1e9
    cq_achieved = nbytes["cq_matvec"] / cq_s / 1e9
    value = world * total_bytes * args.steps / elapsed_s / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(elapsed_s * 1e3 / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded; weights resident in HBM)",
        "config": {"workload": WORKLOAD, "batch": 1,
                   "bytes_per_step": total_bytes,
                   "l2": "inputs larger than L2: each step streams %.2f GB" % (total_bytes / 1e9),
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "streams": "CQ chain (prepare -> matvec, gather) on a second stream beside the F8 head"},
        "us_per_matvec": {k: round(v * 1e3, 3) for k, v in per_kernel_ms.items()},
        "us_per_matvec_note": "event pair around each call in a second timed pass (includes launch latency)",
        "gbs_per_kernel": {k: round(nbytes[k] / (per_kernel_ms[k] / 1e3) / 1e9, 1)
                           for k in names},
        "hbm_frac_of_8tbs": round(value / world / NOMINAL_HBM_GBS, 4),
        "roofline": {"kernel": "f8_matvec (245760x4096, batch 1)", "bound": "hbm",
                     "timing": "%d back-to-back launches between one event pair" % nh,
                     "achieved": round(f8_achieved, 1), "peak": peak,
                     "peak_kind": peak_kind + " copy bandwidth", "unit": "GB/s",
                     "frac": round(f8_achieved / peak, 4), "traffic": ncu_traffic(),
                     "algorithmic_bytes": nbytes["f8_matvec"]},
        "roofline_cq": {"kernel": "cq_matvec (CQ 2-bit 32768x512, input 500, batch 1)",
                        "bound": "hbm",
                        "timing": "CUDA graph of %d back-to-back calls over %d distinct copies "
                                  "(L2-cold), median of 20 replays" % (cq_copies, cq_copies),
                        "achieved": round(cq_achieved, 1), "peak": peak,
                        "peak_kind": peak_kind + " copy bandwidth", "unit": "GB/s",
                        "frac": round(cq_achieved / peak, 4), "traffic": None,
                        "us_per_call": round(cq_s * 1e6, 3),
                        "algorithmic_bytes": nbytes["cq_matvec"]},
        "roofline_head_b8": {"kernel": "f8_matvec (245760x4096, batch 8: tcgen05 kind::f8f6f4, weights by TMA)",
                             "bound": "hbm",
                             "timing": "%d back-to-back launches between one event pair" % n8,
                             "achieved": round(b8_achieved, 1), "peak": peak,
                             "peak_kind": peak_kind + " copy bandwidth", "unit": "GB/s",
                             "frac": round(b8_achieved / peak, 4), "traffic": None,
                             "us_per_call": round(f8_b8_s * 1e6, 2),
                             "algorithmic_bytes": b8_bytes,
                             "ncu": "profiles/f8_tc_head_b8.md (131072 rows: DRAM reads 1.000x the weights, "
                                    "tensor pipe 16%)"},
        "cpu_baseline": cpu,
        "context": {"pages_cpu_figures": PAGES_CPU_CONTEXT,
                    "this_run_head_s_per_token": round(f8_s, 6)},
        "e2e": {"value": round(world * total_bytes * args.steps / e2e_s / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "clocks": clock_info,
        "gpu_launches": 4 * args.steps,
    }
    print(json.dumps(line), flush=True)
    if d is not None:
        d.destroy_process_group()


# --------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and the reference arm)
# --------------------------------------------------------------------------

def oracle_sample(cq, f8, frac, threads):
    """Run the oracle over the first `frac` of the rows of both matrices (plus
    prepare and the full gather); return (seconds, algorithmic bytes)."""
    import oracle
    om = oracle.CQMatrix(cq.output, cq.input, cq.input_padded, cq.group, cq.bits, cq.packed,
                         cq.norms, cq.codebook)
    r3 = max(1, int(cq.output * frac))
    r5 = max(1, int(f8.R * frac))
    t = time.perf_counter()
    p = oracle.cq_prepare(cq.x, cq.input_padded, cq.group, mode="f32")
    om.matvec(p, rows=(0, r3), threads=threads, with_mag=False)
    om.dequantize_rows(cq.rows)
    oracle.f8_matvec(f8.w, f8.scale, f8.x, rows=(0, r5), threads=threads, with_mag=False)
    dt = time.perf_counter() - t
    b = (cq_prepare_bytes(cq.input, cq.input_padded)
         + cq_matvec_bytes(r3, cq.input_padded, cq.group, cq.bits)
         + cq_gather_bytes(len(cq.rows), cq.input, cq.input_padded, cq.group, cq.bits)
         + f8_bytes(r5, f8.C, f8.SR, f8.SC))
    return dt, b, r3, r5


def calibrate(cq, f8, threads, target_s):
    """Fraction of the workload the oracle covers in about target_s seconds."""
    oracle_sample(cq, f8, 1.0 / 8192, threads)  # first call: library load, first touches
    frac = 1.0 / 1024
    for _ in range(8):
        dt, b, r3, r5 = oracle_sample(cq, f8, frac, threads)
        if dt >= 0.2 * target_s or frac >= 1.0:
            break
        frac = min(1.0, frac * 8)
    return min(1.0, frac * target_s / max(dt, 1e-6))


def cpu_baseline(cq, f8, target_s=2.0):
    threads = os.cpu_count() or 1
    frac = calibrate(cq, f8, threads, target_s)
    dt, b, r3, r5 = oracle_sample(cq, f8, frac, threads)
    return {"value": round(b / dt / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": "float64 C oracle, %d threads: prepare + 64-row gather + first %d of 32768 "
                      "CQ rows + first %d of 245760 F8 rows (%.3f%% of the step), %.2f s" % (
                          threads, r3, r5, 100 * frac, dt)}


def run_reference(args):
    world, rank, local = dist_env()
    if world > 1 and rank != 0:
        return
    cq, f8 = make_inputs()
    threads = os.cpu_count() or 1
    frac = calibrate(cq, f8, threads, 1.0)
    for _ in range(args.warmup):
        oracle_sample(cq, f8, frac, threads)
    total_t, total_b = 0.0, 0
    for _ in range(args.steps):
        dt, b, r3, r5 = oracle_sample(cq, f8, frac, threads)
        total_t += dt
        total_b += b
    value = total_b / total_t / 1e9
    sample = ("float64 C oracle, %d threads, per step: prepare + 64-row gather + first %d of "
              "32768 CQ rows + first %d of 245760 F8 rows (%.3f%% of the workload)" % (
                  threads, r3, r5, 100 * frac))
    line = {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_t * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": WORKLOAD, "batch": 1},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample, "sample_fraction": frac},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# per-workload sweep (--configs): every workload and batch of the pages'
# shapes, one JSON line each (the default run prints the one step line)
# --------------------------------------------------------------------------

def _graph_time(torch, calls, reps=20):
    """Median microseconds per call of a CUDA graph holding `calls`."""
    def checked(c):
        def run(sh):
            st = c(sh)
            if st != 0:
                raise RuntimeError("call failed with status %d" % st)
        return run
    calls = [checked(c) for c in calls]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for c in calls[:4]:
            c(s.cuda_stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for c in calls:
            c(s.cuda_stream)
    g.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3 / len(calls))
    return statistics.median(ts), min(ts)


def _cold_single(torch, call, flush, reps=20):
    """Median and best microseconds of one call timed alone: L2 flushed by a
    write larger than it, then an event pair around the single launch."""
    st = torch.cuda.current_stream()
    ts = []
    for _ in range(reps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        if call(st.cuda_stream) != 0:
            raise RuntimeError("call failed")
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3)
    return statistics.median(ts), min(ts)


def oracle_config_lines(only=None):
    """CPU baseline per workload: the oracle's time for one whole C3 matvec
    (CQ 2-bit vocabulary, prepare + matvec) and one whole C4 matvec (F8
    4096 x 4096, batch 1), on one host thread and on all of them."""
    import oracle
    from quantized_weight_matvec_gb300 import synth
    cores = os.cpu_count() or 1
    for name in ("cq2_vocab", "f8_4096"):
        if only and only not in name:
            continue
        if name == "cq2_vocab":
            c = synth.workload_inputs(name, batch=1)
            om = oracle.CQMatrix(c.output, c.input, c.input_padded, c.group, c.bits, c.packed,
                                 c.norms, c.codebook)
            nb = (cq_prepare_bytes(c.input, c.input_padded)
                  + cq_matvec_bytes(c.output, c.input_padded, c.group, c.bits))

            def once(th):
                p = oracle.cq_prepare(c.x, c.input_padded, c.group, mode="f32")
                om.matvec(p, threads=th, with_mag=False)
            op = "oracle cq_prepare + cq_matvec"
        else:
            f = synth.workload_inputs(name, batch=1)
            nb = f8_bytes(f.R, f.C, f.SR, f.SC)

            def once(th):
                oracle.f8_matvec(f.w, f.scale, f.x, threads=th, with_mag=False)
            op = "oracle f8_matvec"
        once(cores)  # library load and first touches
        for th in sorted({1, cores}):
            ts = []
            for _ in range(3):
                t = time.perf_counter()
                once(th)
                ts.append(time.perf_counter() - t)
            us = statistics.median(ts) * 1e6
            print(json.dumps({"workload": name, "batch": 1, "op": op, "bytes": nb,
                              "us_median": round(us, 1), "gbs": round(nb / us / 1e3, 3),
                              "cpu_baseline": {"kind": "oracle", "cores": th}}), flush=True)


def run_configs(args):
    import torch
    from quantized_weight_matvec_gb300 import qmv, synth
    qmv.load()
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    peak, peak_kind = measured_hbm_gbs()
    dev = torch.device("cuda", 0)

    def copies_for(nbytes):
        return max(1, min(4096, -(-2 * l2 // max(nbytes, 1))))

    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)

    def emit(name, batch, op, nbytes, us_med, us_best, ncopies, call=None):
        rec = {"workload": name, "batch": batch, "op": op, "bytes": nbytes,
               "us_median": round(us_med, 3), "us_best": round(us_best, 3),
               "gbs": round(nbytes / us_med / 1e3, 1),
               "frac_of_measured_hbm": round(nbytes / us_med / 1e3 / peak, 4),
               "frac_of_8tbs": round(nbytes / us_med / 1e3 / NOMINAL_HBM_GBS, 4),
               "l2_cold_copies": ncopies}
        if call is not None:  # one call alone after an L2 flush, launch latency included
            cm, cb = _cold_single(torch, call, flush)
            rec["us_single_cold_median"] = round(cm, 3)
            rec["us_single_cold_best"] = round(cb, 3)
        print(json.dumps(rec), flush=True)

    # matrix sets: one activation, several matrices sharing it (needle-2
    # sections 6-7: phiPre/phiPost/phiResidual, Q/K/V).  Per set call, three
    # ways: prepare + one call per matrix, prepare + cq_matvec_multi, and the
    # fused cq_prepare_matvec.
    for label, outs, inp, group, bits in (("set3_2048x512", (2048, 2048, 2048), 512, 64, 2),
                                          ("set3_2048x512", (2048, 2048, 2048), 512, 64, 4),
                                          ("cq2_vocab_fused", (32768,), 500, 128, 2)):
        if args.only and args.only not in label:
            continue
        cs = [synth.cq_inputs(60 + i, o, inp, group, bits, x_scale=3.0) for i, o in enumerate(outs)]
        c0 = cs[0]
        per = [c.output * (c.row_bytes + 2 * (c.input_padded // c.group)) for c in cs]
        k = copies_for(sum(per))
        cb = torch.from_numpy(c0.codebook).to(dev)
        packs = [torch.from_numpy(np.ascontiguousarray(np.broadcast_to(c.packed, (k,) + c.packed.shape))).to(dev)
                 for c in cs]
        norms = [torch.from_numpy(np.ascontiguousarray(np.broadcast_to(c.norms.view(np.int16), (k,) + c.norms.shape))).to(dev)
                 for c in cs]
        sets = [[qmv.CQMatrix(c.output, c.input, c.input_padded, c.group, c.bits, packs[j][i],
                              norms[j][i], cb) for j, c in enumerate(cs)] for i in range(k)]
        x = torch.from_numpy(c0.x).to(dev)
        p = torch.empty((1, c0.input_padded), device=dev)
        ys = [torch.empty((1, c.output), device=dev) for c in cs]
        yp = [y.data_ptr() for y in ys]
        nb = cq_prepare_bytes(c0.input, c0.input_padded) + sum(
            cq_matvec_bytes(c.output, c.input_padded, c.group, c.bits) for c in cs)

        def sep(ms):
            def run(sh):
                st = qmv.cq_prepare(ms[0].struct, x.data_ptr(), 1, p.data_ptr(), sh)
                for m, y in zip(ms, yp):
                    st = st or qmv.cq_matvec(m.struct, p.data_ptr(), 1, y, sh)
                return st
            return run

        def multi(ms):
            def run(sh):
                return (qmv.cq_prepare(ms[0].struct, x.data_ptr(), 1, p.data_ptr(), sh) or
                        qmv.cq_matvec_multi([m.struct for m in ms], p.data_ptr(), 1, yp, sh))
            return run

        def fused(ms):
            return lambda sh: qmv.cq_prepare_matvec([m.struct for m in ms], x.data_ptr(), 1, 0, yp, sh)

        tag = "%s/%dbit" % (label, bits)
        for op, mk in (("prepare+cq_matvec x%d" % len(cs), sep),
                       ("prepare+cq_matvec_multi", multi), ("cq_prepare_matvec", fused)):
            med, best = _graph_time(torch, [mk(ms) for ms in sets])
            emit(tag, 1, op, nb, med, best, k)
        del packs, norms, sets

    for name, wl in synth.WORKLOADS.items():
        if args.only and args.only not in name:
            continue
        for batch in wl["batch"]:
            if wl["kind"] == "cq":
                for bits in wl["bits"]:
                    c = synth.workload_inputs(name, bits=bits, batch=batch)
                    nb = cq_matvec_bytes(c.output, c.input_padded, c.group, c.bits, batch)
                    k = copies_for(c.output * (c.row_bytes + 2 * (c.input_padded // c.group)))
                    packed = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(
                        c.packed, (k,) + c.packed.shape))).to(dev)
                    norms = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(
                        c.norms.view(np.int16), (k,) + c.norms.shape))).to(dev)
                    cb = torch.from_numpy(c.codebook).to(dev)
                    mats = [qmv.CQMatrix(c.output, c.input, c.input_padded, c.group, c.bits,
                                         packed[i], norms[i], cb) for i in range(k)]
                    x = torch.from_numpy(c.x).to(dev)
                    p = qmv.cq_prepare_t(mats[0], x)
                    y = torch.empty((batch, c.output), device=dev)
                    calls = [(lambda m: lambda sh: qmv.cq_matvec(m.struct, p.data_ptr(), batch,
                                                                  y.data_ptr(), sh))(m)
                             for m in mats]
                    med, best = _graph_time(torch, calls)
                    emit("%s/%dbit" % (name, bits), batch, "cq_matvec", nb, med, best, k,
                         call=calls[0])
                    pc = [lambda sh: qmv.cq_prepare(mats[0].struct, x.data_ptr(), batch,
                                                    p.data_ptr(), sh)] * 64
                    med, best = _graph_time(torch, pc)
                    emit("%s/%dbit" % (name, bits), batch, "cq_prepare",
                         cq_prepare_bytes(c.input, c.input_padded, batch), med, best, 1,
                         call=pc[0])
                    if wl.get("gather"):
                        ids = torch.from_numpy(c.rows).to(dev)
                        emb = torch.empty((len(c.rows), c.input), device=dev)
                        gc = [(lambda m: lambda sh: qmv.cq_dequantize_row(
                            m.struct, ids.data_ptr(), ids.numel(), emb.data_ptr(), 0, sh))(m)
                            for m in mats]
                        med, best = _graph_time(torch, gc)
                        emit("%s/%dbit" % (name, bits), len(c.rows), "cq_dequantize_row",
                             cq_gather_bytes(len(c.rows), c.input, c.input_padded, c.group,
                                             c.bits), med, best, k, call=gc[0])
                    del packed, norms, mats
            elif wl["kind"] == "hmlp":
                f = synth.workload_inputs(name, batch=batch)
                # x, residual, u in and out: 4 [batch, n] float32; three diagonals
                nb = 4 * (4 * batch * f.n + 3 * f.D)
                hx, hr, hu = (torch.from_numpy(a).to(dev) for a in (f.x, f.residual, f.u))
                hd = [torch.from_numpy(a).to(dev) for a in (f.d1, f.d2, f.d3)]
                ho = torch.empty((batch, f.n), device=dev)
                hcalls = [lambda sh: qmv.hadamard_mlp(
                    hx.data_ptr(), f.n, f.D, hd[0].data_ptr(), hd[1].data_ptr(), hd[2].data_ptr(),
                    hr.data_ptr(), hu.data_ptr(), batch, ho.data_ptr(), sh)] * 64
                med, best = _graph_time(torch, hcalls)
                emit("%s/D%d" % (name, f.D), batch, "hadamard_mlp", nb, med, best, 1,
                     call=hcalls[0])
            elif wl["kind"] == "i8":
                f = synth.workload_inputs(name, batch=batch)
                nb = f.R * f.C + f.R * ((f.C + 15) // 16) + 4 * batch * (f.C + f.R)
                k = copies_for(f.R * f.C)
                w = torch.from_numpy(f.w).to(dev)
                ws = [w] + [w.clone() for _ in range(k - 1)]
                s8 = torch.from_numpy(f.scale).to(dev)
                x = torch.from_numpy(f.x).to(dev)
                y = torch.empty((batch, f.R), device=dev)
                calls = [(lambda wi: lambda sh: qmv.i8_matvec(
                    wi.data_ptr(), f.R, f.C, s8.data_ptr(), x.data_ptr(), batch, y.data_ptr(),
                    sh))(wi) for wi in ws]
                if k == 1:
                    calls = calls * 8
                med, best = _graph_time(torch, calls, reps=10)
                emit(name, batch, "i8_matvec", nb, med, best, k, call=calls[0])
                # int8 activations with per-32 scales (Mnemonic "In the
                # browser"): the quantizer, then the int8 x int8 matvec
                xq, xsc = qmv.i8_quantize_x_t(x)
                xg = (f.C + 31) // 32
                qc = [lambda sh: qmv.i8_quantize_x(x.data_ptr(), f.C, batch, xq.data_ptr(),
                                                   xsc.data_ptr(), sh)] * 64
                med, best = _graph_time(torch, qc)
                emit(name, batch, "i8_quantize_x", batch * (5 * f.C + 4 * xg), med, best, 1,
                     call=qc[0])
                nbq = f.R * f.C + f.R * ((f.C + 15) // 16) + batch * (f.C + 4 * xg) + 4 * batch * f.R
                qcalls = [(lambda wi: lambda sh: qmv.i8_matvec_q8(
                    wi.data_ptr(), f.R, f.C, s8.data_ptr(), xq.data_ptr(), xsc.data_ptr(), batch,
                    y.data_ptr(), sh))(wi) for wi in ws]
                if k == 1:
                    qcalls = qcalls * 8
                med, best = _graph_time(torch, qcalls, reps=10)
                emit(name, batch, "i8_matvec_q8", nbq, med, best, k, call=qcalls[0])
                # the I8 head then top-64 temperature sampling (logits stored)
                tk = 64
                wst = torch.empty(qmv.TOPK_WORKSPACE_BYTES, dtype=torch.uint8, device=dev)
                uu = torch.rand(batch, device=dev)
                ti = torch.empty((batch, tk), dtype=torch.int64, device=dev)
                tv = torch.empty((batch, tk), device=dev)
                tp = torch.empty((batch, tk), device=dev)
                tt = torch.empty(batch, dtype=torch.int64, device=dev)
                tcalls = [(lambda wi: lambda sh: qmv.i8_matvec_topk_sample(
                    wi.data_ptr(), f.R, f.C, s8.data_ptr(), x.data_ptr(), batch, y.data_ptr(), tk,
                    1.0, uu.data_ptr(), ti.data_ptr(), tv.data_ptr(), tp.data_ptr(),
                    tt.data_ptr(), wst.data_ptr(), wst.numel(), sh))(wi) for wi in ws]
                if k == 1:
                    tcalls = tcalls * 8
                med, best = _graph_time(torch, tcalls, reps=10)
                emit(name, batch, "i8_matvec_topk_sample(k=64)", nb + batch * (4 + tk * 16 + 8),
                     med, best, k, call=tcalls[0])
                del ws, w
            else:
                f = synth.workload_inputs(name, batch=batch)
                nb = f8_bytes(f.R, f.C, f.SR, f.SC, batch)
                k = copies_for(f.R * f.C)
                w = torch.from_numpy(f.w).to(dev)
                ws = [w] + [w.clone() for _ in range(k - 1)]
                s5 = torch.from_numpy(f.scale).to(dev)
                x = torch.from_numpy(f.x).to(dev)
                y = torch.empty((batch, f.R), device=dev)
                calls = [(lambda wi: lambda sh: qmv.f8_matvec(
                    wi.data_ptr(), f.R, f.C, s5.data_ptr(), f.SR, f.SC, x.data_ptr(), batch,
                    y.data_ptr(), sh))(wi) for wi in ws]
                if k == 1:
                    calls = calls * 8
                med, best = _graph_time(torch, calls, reps=10)
                emit(name, batch, "f8_matvec", nb, med, best, k, call=calls[0])
                # head + greedy selection (no logits stored)
                wsp = torch.zeros(qmv.f8_argmax_workspace_bytes(batch), dtype=torch.uint8,
                                  device=dev)
                oi = torch.empty(batch, dtype=torch.int64, device=dev)
                ov = torch.empty(batch, device=dev)
                acalls = [(lambda wi: lambda sh: qmv.f8_matvec_argmax(
                    wi.data_ptr(), f.R, f.C, s5.data_ptr(), f.SR, f.SC, x.data_ptr(), batch, 0,
                    oi.data_ptr(), ov.data_ptr(), wsp.data_ptr(), wsp.numel(), sh))(wi)
                    for wi in ws]
                if k == 1:
                    acalls = acalls * 8
                med, best = _graph_time(torch, acalls, reps=10)
                emit(name, batch, "f8_matvec_argmax", nb - 4 * batch * f.R + 12 * batch, med,
                     best, k, call=acalls[0])
                if batch > 4:  # no y, but room for the logits in the workspace (tcgen05 at 5..8)
                    wbig = torch.zeros(qmv.f8_argmax_workspace_bytes(batch, f.R), dtype=torch.uint8,
                                       device=dev)
                    bcalls = [(lambda wi: lambda sh: qmv.f8_matvec_argmax(
                        wi.data_ptr(), f.R, f.C, s5.data_ptr(), f.SR, f.SC, x.data_ptr(), batch, 0,
                        oi.data_ptr(), ov.data_ptr(), wbig.data_ptr(), wbig.numel(), sh))(wi)
                        for wi in ws]
                    if k == 1:
                        bcalls = bcalls * 8
                    med, best = _graph_time(torch, bcalls, reps=10)
                    emit(name, batch, "f8_matvec_argmax(logits in workspace)", nb + 12 * batch, med,
                         best, k, call=bcalls[0])
                    del wbig
                if batch > 1:  # logits stored too: the batch 5..8 head then runs on tcgen05
                    ycalls = [(lambda wi: lambda sh: qmv.f8_matvec_argmax(
                        wi.data_ptr(), f.R, f.C, s5.data_ptr(), f.SR, f.SC, x.data_ptr(), batch,
                        y.data_ptr(), oi.data_ptr(), ov.data_ptr(), wsp.data_ptr(), wsp.numel(),
                        sh))(wi) for wi in ws]
                    if k == 1:
                        ycalls = ycalls * 8
                    med, best = _graph_time(torch, ycalls, reps=10)
                    emit(name, batch, "f8_matvec_argmax(y stored)", nb + 12 * batch, med, best, k,
                         call=ycalls[0])
                # head + top-64 temperature sampling (logits stored)
                tk = 64
                wst = torch.empty(qmv.TOPK_WORKSPACE_BYTES, dtype=torch.uint8, device=dev)
                uu = torch.rand(batch, device=dev)
                ti = torch.empty((batch, tk), dtype=torch.int64, device=dev)
                tv = torch.empty((batch, tk), device=dev)
                tp = torch.empty((batch, tk), device=dev)
                tt = torch.empty(batch, dtype=torch.int64, device=dev)
                tcalls = [(lambda wi: lambda sh: qmv.f8_matvec_topk_sample(
                    wi.data_ptr(), f.R, f.C, s5.data_ptr(), f.SR, f.SC, x.data_ptr(), batch,
                    y.data_ptr(), tk, 1.0, uu.data_ptr(), ti.data_ptr(), tv.data_ptr(),
                    tp.data_ptr(), tt.data_ptr(), wst.data_ptr(), wst.numel(), sh))(wi)
                    for wi in ws]
                if k == 1:
                    tcalls = tcalls * 8
                med, best = _graph_time(torch, tcalls, reps=10)
                emit(name, batch, "f8_matvec_topk_sample(k=64)",
                     nb + batch * (4 + tk * 16 + 8), med, best, k, call=tcalls[0])
                del ws, w
    oracle_config_lines(args.only)


# --------------------------------------------------------------------------
# one kernel on a small case, for ncu captures (--case): no timings are
# printed, since numbers taken under a profiler are not measurements
# --------------------------------------------------------------------------

def run_case(args):
    """Run one kernel of the path --iters times on a seeded synthetic case
    and print a checksum.  Cases: f8 (E4M3 rows x 4096, scales [rows/128,
    32]), f8am (the same with greedy selection), i8 (int8 rows x 4096,
    per-16 E8M0 scales), i8q (the same weights x int8 activations), cq2
    (2-bit rows x 512, input 500, group 128: the table kernel), cqvec
    (--bits-bit rows x 512, group 64: the vectorised kernel), gather (64 rows
    of a 32768 x 512 2-bit matrix), prepare, topk (top-64 temperature
    sampling over --rows normal logits per vector)."""
    import torch
    from quantized_weight_matvec_gb300 import qmv, synth
    qmv.load()
    dev = torch.device("cuda", 0)
    k, rows, batch = args.case, args.rows, args.batch
    if k in ("f8", "f8am"):
        f = synth.f8_inputs(5, rows, 4096, max(1, rows // 128), 32, 118, 132, batch=batch)
        w, s, x = (torch.from_numpy(a).to(dev) for a in (f.w, f.scale, f.x))
        y = torch.empty((batch, rows), device=dev)
        for _ in range(args.iters):
            if k == "f8":
                qmv.f8_matvec_t(w, s, x, out=y)
            else:
                qmv.f8_matvec_argmax_t(w, s, x, y=y)
        out = y
    elif k in ("i8", "i8q"):
        f = synth.i8_inputs(7, rows, 4096, 110, 124, batch=batch)
        w, s, x = (torch.from_numpy(a).to(dev) for a in (f.w, f.scale, f.x))
        y = torch.empty((batch, rows), device=dev)
        xq, xs = qmv.i8_quantize_x_t(x)
        for _ in range(args.iters):
            if k == "i8":
                qmv.i8_matvec_t(w, s, x, out=y)
            else:
                qmv.i8_matvec_q8_t(w, s, xq, xs, out=y)
        out = y
    elif k == "topk":
        g = torch.Generator(device="cpu").manual_seed(0)
        y = (torch.randn((batch, rows), generator=g) * 3).to(dev)
        u = torch.rand(batch, generator=g).to(dev)
        for _ in range(args.iters):
            idx, val, prob, tok = qmv.topk_sample_t(y, 64, 1.0, u)
        out = prob
    elif k == "cqvec":
        c = synth.cq_inputs(2, rows, 512, 64, args.bits, batch=batch)
        m = qmv.CQMatrix.from_numpy(c, device=dev)
        p = qmv.cq_prepare_t(m, torch.from_numpy(c.x).to(dev))
        for _ in range(args.iters):
            out = qmv.cq_matvec_t(m, p)
    else:
        n = rows if k == "cq2" else 32768
        c = synth.cq_inputs(3, n, 500, 128, 2, batch=batch, x_scale=3.0, gather=64)
        m = qmv.CQMatrix.from_numpy(c, device=dev)
        x = torch.from_numpy(c.x).to(dev)
        p = qmv.cq_prepare_t(m, x)
        for _ in range(args.iters):
            if k == "cq2":
                out = qmv.cq_matvec_t(m, p)
            elif k == "gather":
                out = qmv.cq_dequantize_row_t(m, torch.from_numpy(c.rows).to(dev))
            else:
                out = qmv.cq_prepare_t(m, x, out=p)
    torch.cuda.synchronize()
    print("checksum %.6e" % float(out.double().abs().sum()))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--configs", action="store_true",
                    help="per-workload sweep (one JSON line per workload, batch and op)")
    ap.add_argument("--only", default="",
                    help="with --configs: only the workloads whose name contains this text")
    ap.add_argument("--case", choices=["f8", "f8am", "i8", "i8q", "cq2", "cqvec", "gather",
                                       "prepare", "topk"],
                    help="run one kernel on a small case for an ncu capture (no timings)")
    ap.add_argument("--rows", type=int, default=65536, help="with --case: matrix rows")
    ap.add_argument("--bits", type=int, default=4, help="with --case cqvec: index width")
    ap.add_argument("--batch", type=int, default=1, help="with --case: activation vectors")
    ap.add_argument("--iters", type=int, default=3, help="with --case: calls")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    if args.case:
        run_case(args)
    elif args.configs:
        run_configs(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
