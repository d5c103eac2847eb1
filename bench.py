#!/usr/bin/env python3
"""Benchmark of the THD zigzag <-> contiguous layout conversion on one GB300.

A step is one pass of the hot path over one packed microbatch: zigzag
partition indices, the route in both directions (validation, interval
counts, identity flags), then every simulated layer's swap pair
(zigzag->contiguous, contiguous->zigzag) on the hidden states.  The default
workload is the log-normal 128K-token packing with cp=4 and 4 KiB rows
(x bf16 [131072, 16, 128]) reused by 48 layers; the working set (1 GiB in
+ 1 GiB out ping-pong) is far larger than L2, so no flush is needed.

value      = swap payload bytes (2 * T * row_bytes per swap, read + write)
             per second of whole-step device time, max over ranks.
e2e        = the same with the step's input copied host->device from pinned
             memory and the result copied back inside the timed region.
roofline   = the swap kernel alone: payload bytes per launch / its average
             launch time, against the measured copy bandwidth.
cpu_baseline / --impl reference = the CPU oracle on a bounded sample.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl thd|reference]
    torchrun --nproc-per-node N bench.py --gpus N ...   (one rank per GPU,
    independent microbatches: weak scaling, no collective on the data path)
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402
import torch.distributed as dist  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "THD zigzag<->contiguous swap HBM GB/s & % of peak; route-build µs per microbatch"
SPEC_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def parse_args():
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["thd", "reference"], default="thd")
    p.add_argument("--workload", default="lognorm128k", choices=[w.name for w in W.WORKLOADS])
    p.add_argument("--layers", type=int, default=None, help="swap pairs per step (default: 48; pipeline 1)")
    p.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle work for cpu_baseline")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--cp-exchange", action="store_true",
                   help="one CP rank per GPU (--gpus = the workload's cp): the conversion between GPUs, "
                        "per-rank pack -> NCCL all-to-all -> per-rank scatter, instead of independent replicas")
    p.add_argument("--only-prep-at-scale", action="store_true",
                   help="run only the data-preparation kernels at 16.8 M tokens and print their timings")
    p.add_argument("--no-other-configs", action="store_true",
                   help="skip the swap / route timings of the other full-size workloads")
    return p.parse_args()


# ---------------------------------------------------------------------------
# environment
# ---------------------------------------------------------------------------

def setup_dist(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world, device=None):
    if world > 1:
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(value: float, world: int, device) -> float:
    """Largest value over all ranks (elapsed times: the slowest rank decides)."""
    if world == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int, device) -> float:
    if world == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def copy_engine_digest():
    """sha256 of the swap kernel's sources: copy.cu followed by tma.cuh."""
    h = hashlib.sha256()
    for name in ("copy.cu", "tma.cuh"):
        with open(os.path.join(ROOT, "context_packed_sequence_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def swap_traffic_record(workload: str):
    """dram bytes per swap launch on this workload from the committed ncu
    summary (profiles/bulk_copy_swap_<workload>.md), or None when the summary
    is missing or the copy kernel's sources changed since."""
    path = os.path.join(ROOT, "profiles", f"bulk_copy_swap_{workload}.md")
    try:
        text = open(path).read()
        digest = copy_engine_digest()
    except OSError:
        return None
    fields = {}
    for line in text.splitlines():
        if line.startswith("- ") and ":" in line:
            k, v = line[2:].split(":", 1)
            fields[k.strip()] = v.strip()
    recorded = next((v.strip("`") for k, v in fields.items() if k.startswith("copy engine sha256")), None)
    if recorded != digest:
        return None
    try:
        return int(fields["dram bytes per launch"].split()[0].replace(",", ""))
    except (KeyError, ValueError, IndexError):
        return None


def plan_kernel_name(row_bytes: int) -> str:
    """The kernel thd_swap launches for this row size (the plans in copy.cu)."""
    if row_bytes % 16:
        return "copy_rows_kernel<unit, SwapMap, false> (thd_swap)"
    if row_bytes < 208:
        fit = 8192 // (32 * row_bytes)
        k = 16 if fit >= 16 else 8 if fit >= 8 else 4 if fit >= 4 else 2 if fit >= 2 else 1
        return f"run_copy_kernel<{k}, {2 if 32 * k * row_bytes >= 8192 else 3}, SwapMap, false> (thd_swap)"
    nst = 2 if row_bytes <= 8192 else (4 if row_bytes <= 16384 else (3 if row_bytes <= 32768 else 4))
    return f"bulk_copy_kernel<{nst}, SwapMap, false> (thd_swap)"


def smi_gpu_id(device) -> str:
    """The nvidia-smi id of a CUDA device: its PCI address, which does not
    depend on CUDA_VISIBLE_DEVICES; else its index mapped through that list."""
    try:
        p = torch.cuda.get_device_properties(device)
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except (AttributeError, RuntimeError, AssertionError):
        pass
    ids = [v.strip() for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    if device.index is not None and device.index < len(ids):
        return ids[device.index]
    return str(device.index or 0)


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    QUERY = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.out = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.seek(0)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[3:7]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# inputs
# ---------------------------------------------------------------------------

def make_inputs(w, device, rank):
    """(cu list, T, raw tokens or None) of the workload; x is drawn separately."""
    if w.name == "pipeline":
        raw = W.raw_pipeline_tokens(w.seed + 1000 * rank)
        return None, None, raw
    cu = W.boundaries(W.doc_lengths(w.name))
    return cu, cu[-1], None


# ---------------------------------------------------------------------------
# timing helpers (CUDA events on the launching stream)
# ---------------------------------------------------------------------------

def single_us(fn, stream, device, reps=30, skip=10):
    """Median duration of one launch between two CUDA events, the GPU kept
    busy ahead of it so host launch latency is not counted."""
    ts = []
    for it in range(reps):
        torch.cuda._sleep(200_000)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize(device)
        if it >= skip:
            ts.append(a.elapsed_time(b) * 1e3)
    return round(statistics.median(ts), 2)


def back_to_back_us(fn, stream, device, launches=20, reps=12, skip=2):
    """Per-launch duration of `launches` launches back to back between two
    CUDA events (each launch waits for the one before, so launch latency
    overlaps the previous launch), median over reps."""
    ts = []
    for it in range(reps):
        torch.cuda._sleep(200_000)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(launches):
            fn()
        b.record(stream)
        torch.cuda.synchronize(device)
        if it >= skip:
            ts.append(a.elapsed_time(b) * 1e3 / launches)
    return round(statistics.median(ts), 2)


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

def run_thd(args, rank, world, local):
    import context_packed_sequence_gb300 as thd
    from context_packed_sequence_gb300 import _lib as L
    import ctypes

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    w = W.BY_NAME[args.workload]
    layers = args.layers if args.layers is not None else (1 if w.name == "pipeline" else 48)
    cp = w.cp
    stream = torch.cuda.current_stream(device)
    sp = stream.cuda_stream
    lib = L.load()

    cu_list, T, raw = make_inputs(w, device, rank)
    status = thd.new_status(device)
    extra = None
    if raw is not None:
        raw_d = torch.from_numpy(raw).to(device)
        B, S = raw.shape
        tok, cu_v, cu_d = thd.pack_docs(raw_d, W.EOD_ID, 2 * cp, pad_id=0)   # data prep, untimed
        T = int(tok.numel())
        n_docs = cu_d.numel() - 1
        cap_tok, cap_docs = B * S * 2 * cp, B * S + 1
        ptok = torch.empty(cap_tok, dtype=torch.int32, device=device)
        pcu_v = torch.empty(cap_docs, dtype=torch.int32, device=device)
        pcu = torch.empty(cap_docs, dtype=torch.int32, device=device)
        counts = torch.zeros(2, dtype=torch.int64, device=device)
        ws = torch.empty(lib.thd_pack_docs_workspace_bytes(B, S), dtype=torch.uint8, device=device)
        labels = torch.empty((w.mtp_depth + 1, T), dtype=torch.int32, device=device)
        lmask = torch.empty((w.mtp_depth + 1, T), dtype=torch.uint8, device=device)
        valid = torch.empty((T,), dtype=torch.uint8, device=device)
        extra = dict(raw=raw_d, B=B, S=S, ptok=ptok, pcu_v=pcu_v, pcu=pcu, counts=counts, ws=ws,
                     labels=labels, lmask=lmask, valid=valid, cap_tok=cap_tok, cap_docs=cap_docs)
    else:
        cu_d = torch.tensor(cu_list, dtype=torch.int32, device=device)
        n_docs = len(cu_list) - 1
    row_bytes = w.row_bytes
    x = W.payload_device(w.seed + 1000 * rank, T, w.hidden, device)
    y = torch.empty_like(x)
    fwd, bwd = thd.Route.pair(T, cp, device)   # one buffer, the common arrays shared
    pidx = torch.empty((cp, T // cp), dtype=torch.int32, device=device)
    swap_bytes = 2 * T * row_bytes
    launches_per_step = 2 + 2 * layers + (3 if extra is not None else 0)

    def front(s):
        """Everything before the swaps: (packing and labels,) partition, routes."""
        if extra is not None:
            e = extra
            lib.thd_pack_docs(e["raw"].data_ptr(), e["B"], e["S"], W.EOD_ID, 0, 0, 2 * cp, 0, None,
                              e["ptok"].data_ptr(), e["cap_tok"], e["pcu_v"].data_ptr(), e["pcu"].data_ptr(), None,
                              None, e["cap_docs"],
                              e["counts"].data_ptr(), e["ws"].data_ptr(), e["ws"].numel(), status.data_ptr(), s)
            lib.thd_roll_labels(e["ptok"].data_ptr(), e["pcu_v"].data_ptr(), e["pcu"].data_ptr(), n_docs, T,
                                w.mtp_depth, 0, None, None, e["labels"].data_ptr(), e["lmask"].data_ptr(),
                                e["valid"].data_ptr(), status.data_ptr(), s)
        lib.thd_partition_indices(cu_d.data_ptr(), n_docs, T, cp, -1, pidx.data_ptr(), status.data_ptr(), s)
        lib.thd_route_build_pair(cu_d.data_ptr(), n_docs, T, cp, ctypes.byref(fwd.c), ctypes.byref(bwd.c),
                                 status.data_ptr(), s)

    def swaps(s, a, b):
        for _ in range(layers):
            lib.thd_swap(a.data_ptr(), b.data_ptr(), row_bytes, ctypes.byref(fwd.c), status.data_ptr(), s)
            lib.thd_swap(b.data_ptr(), a.data_ptr(), row_bytes, ctypes.byref(bwd.c), status.data_ptr(), s)

    # warm-up
    for _ in range(args.warmup):
        front(sp)
        swaps(sp, x, y)
    torch.cuda.synchronize(device)
    code = thd.status_read(status)
    if code != 0:
        raise RuntimeError(f"device status {code} after warm-up")

    # timed region
    n_ev = args.steps
    ev_step = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev + 1)]
    ev_sw = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_ev)]
    clocks = ClockSampler(smi_gpu_id(device)).start() if rank == 0 else None
    barrier(world, device)
    torch.cuda.synchronize(device)
    ev_step[0].record(stream)
    for i in range(n_ev):
        front(sp)
        ev_sw[i][0].record(stream)
        swaps(sp, x, y)
        ev_sw[i][1].record(stream)
        ev_step[i + 1].record(stream)
    torch.cuda.synchronize(device)
    barrier(world, device)
    clock_rec = clocks.stop() if clocks is not None else None
    step_ms_local = ev_step[0].elapsed_time(ev_step[-1])
    per_step_swap_ms = [a.elapsed_time(b) for a, b in ev_sw]
    swap_ms_total = sum(per_step_swap_ms)
    code = thd.status_read(status)
    if code != 0:
        raise RuntimeError(f"device status {code} in the timed region")

    total_ms = max_over_ranks(step_ms_local, world, device)
    bytes_all = sum_over_ranks(float(swap_bytes * 2 * layers * n_ev), world, device)
    value = bytes_all / (total_ms / 1e3) / 1e9
    swap_us = swap_ms_total * 1e3 / (2 * layers * n_ev)
    achieved = swap_bytes / (swap_us * 1e-6) / 1e9
    # per-step average swap time: its median and 10th / 90th percentiles
    per_swap = sorted(v * 1e3 / (2 * layers) for v in per_step_swap_ms)

    def pct(q):
        return round(per_swap[min(len(per_swap) - 1, int(q * (len(per_swap) - 1) + 0.5))], 2)

    swap_dist = {"median": pct(0.5), "p10": pct(0.1), "p90": pct(0.9), "unit": "us per launch",
                 "over": f"{n_ev} steps of {2 * layers} launches"}

    # route build alone: CUDA events around each build, the GPU kept busy so
    # host launch latency is not counted; median of 50
    rb = {"both_directions": [], "zigzag_to_contiguous": [], "contiguous_to_zigzag": [], "partition": []}
    for it in range(60):
        torch.cuda._sleep(200_000)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        ev[0].record(stream)
        lib.thd_route_build_pair(cu_d.data_ptr(), n_docs, T, cp, ctypes.byref(fwd.c), ctypes.byref(bwd.c),
                                 status.data_ptr(), sp)
        ev[1].record(stream)
        lib.thd_route_build(cu_d.data_ptr(), n_docs, T, cp, 0, ctypes.byref(fwd.c), status.data_ptr(), sp)
        ev[2].record(stream)
        lib.thd_route_build(cu_d.data_ptr(), n_docs, T, cp, 1, ctypes.byref(bwd.c), status.data_ptr(), sp)
        ev[3].record(stream)
        lib.thd_partition_indices(cu_d.data_ptr(), n_docs, T, cp, -1, pidx.data_ptr(), status.data_ptr(), sp)
        ev[4].record(stream)
        torch.cuda.synchronize(device)
        if it >= 10:
            for k, name in enumerate(rb):
                rb[name].append(ev[k].elapsed_time(ev[k + 1]) * 1e3)
    route_us = {k: round(statistics.median(v), 2) for k, v in rb.items()}
    route_us["method"] = "median of 50, CUDA events with the GPU kept busy ahead of each launch"

    # The same kernels' own duration: 20 launches back to back between two
    # events (each waits for the previous one, so launch latency overlaps
    # the previous launch), per launch, median of 20.  Single-launch events
    # move in steps of about 2 us on this GPU; this figure resolves below that.
    calls = {
        "both_directions": lambda: lib.thd_route_build_pair(cu_d.data_ptr(), n_docs, T, cp, ctypes.byref(fwd.c),
                                                            ctypes.byref(bwd.c), status.data_ptr(), sp),
        "zigzag_to_contiguous": lambda: lib.thd_route_build(cu_d.data_ptr(), n_docs, T, cp, 0, ctypes.byref(fwd.c),
                                                            status.data_ptr(), sp),
        "contiguous_to_zigzag": lambda: lib.thd_route_build(cu_d.data_ptr(), n_docs, T, cp, 1, ctypes.byref(bwd.c),
                                                            status.data_ptr(), sp),
        "partition": lambda: lib.thd_partition_indices(cu_d.data_ptr(), n_docs, T, cp, -1, pidx.data_ptr(),
                                                       status.data_ptr(), sp),
    }
    b2b = {name: [] for name in calls}
    for it in range(23):
        for name, fn in calls.items():
            torch.cuda._sleep(200_000)
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ev0.record(stream)
            for _ in range(20):
                fn()
            ev1.record(stream)
            torch.cuda.synchronize(device)
            if it >= 3:
                b2b[name].append(ev0.elapsed_time(ev1) * 1e3 / 20)
    route_us["back_to_back"] = {k: round(statistics.median(v), 2) for k, v in b2b.items()}
    route_us["back_to_back_method"] = "20 launches between two CUDA events, per launch, median of 20"

    # packing and labels alone (pipeline workload): CUDA events, median of 20
    prep = None
    if extra is not None:
        e = extra

        def pack_call():
            lib.thd_pack_docs(e["raw"].data_ptr(), e["B"], e["S"], W.EOD_ID, 0, 0, 2 * cp, 0, None,
                              e["ptok"].data_ptr(), e["cap_tok"], e["pcu_v"].data_ptr(), e["pcu"].data_ptr(), None,
                              None, e["cap_docs"],
                              e["counts"].data_ptr(), e["ws"].data_ptr(), e["ws"].numel(), status.data_ptr(), sp)

        def labels_call():
            lib.thd_roll_labels(e["ptok"].data_ptr(), e["pcu_v"].data_ptr(), e["pcu"].data_ptr(), n_docs, T,
                                w.mtp_depth, 0, None, None, e["labels"].data_ptr(), e["lmask"].data_ptr(),
                                e["valid"].data_ptr(), status.data_ptr(), sp)

        def time_call(fn):
            ts = []
            for it in range(30):
                torch.cuda._sleep(200_000)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                torch.cuda.synchronize(device)
                if it >= 10:
                    ts.append(a.elapsed_time(b) * 1e3)
            return statistics.median(ts)

        peak_gbs, _ = measured_peak()
        raw_tokens = e["B"] * e["S"]
        pack_bytes = 4 * raw_tokens + 4 * T + 8 * (n_docs + 1)            # read raw once, write tokens + bounds
        lab_bytes = 4 * T + 8 * (n_docs + 1) + (w.mtp_depth + 1) * 5 * T + T  # tokens in; labels, masks, valid out

        def labels_zz_call():
            lib.thd_roll_labels_zigzag(e["ptok"].data_ptr(), e["pcu_v"].data_ptr(), e["pcu"].data_ptr(), n_docs, T,
                                       cp, w.mtp_depth, 0, None, None, e["labels"].data_ptr(), e["lmask"].data_ptr(),
                                       e["valid"].data_ptr(), status.data_ptr(), sp)

        def b2b_call(fn):
            # the kernels' own duration: 20 launches between two events, per launch
            ts = []
            for it in range(12):
                torch.cuda._sleep(200_000)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for _ in range(20):
                    fn()
                b.record(stream)
                torch.cuda.synchronize(device)
                if it >= 2:
                    ts.append(a.elapsed_time(b) * 1e3 / 20)
            return round(statistics.median(ts), 2)

        pack_us, lab_us, labz_us = time_call(pack_call), time_call(labels_call), time_call(labels_zz_call)
        prep = {
            "method": "us: median of 20 single launches between CUDA events; us_back_to_back: 20 launches "
                      "back to back, per launch, median of 10",
            "pack_docs": {"us": round(pack_us, 2), "us_back_to_back": b2b_call(pack_call), "algorithmic_bytes": pack_bytes,
                          "gbs": round(pack_bytes / pack_us / 1e3, 1),
                          "frac_of_measured": round(pack_bytes / pack_us / 1e3 / peak_gbs, 4)},
            "roll_labels": {"us": round(lab_us, 2), "us_back_to_back": b2b_call(labels_call),
                            "algorithmic_bytes": lab_bytes, "mtp_depth": w.mtp_depth,
                            "gbs": round(lab_bytes / lab_us / 1e3, 1),
                            "frac_of_measured": round(lab_bytes / lab_us / 1e3 / peak_gbs, 4)},
            "roll_labels_zigzag": {"us": round(labz_us, 2), "us_back_to_back": b2b_call(labels_zz_call),
                                   "algorithmic_bytes": lab_bytes, "cp_size": cp,
                                   "gbs": round(lab_bytes / labz_us / 1e3, 1),
                                   "frac_of_measured": round(lab_bytes / labz_us / 1e3 / peak_gbs, 4)},
        }
        if thd.status_read(status) != 0:
            raise RuntimeError("device status set while timing packing / labels")

    # Ulysses exchange of the same hidden states (each token row = cp head groups)
    uly = None
    if row_bytes % cp == 0 and T % cp == 0:
        def uly_time(direction, src, dst):
            """Per-launch time of 20 launches back to back (as the swaps run
            inside a step), median of 10: each direction rewrites the same
            output, head -> sequence of y giving back x."""
            ts = []
            for it in range(12):
                torch.cuda._sleep(200_000)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for _ in range(20):
                    lib.thd_ulysses_swap(src.data_ptr(), dst.data_ptr(), T, cp, row_bytes, direction,
                                         status.data_ptr(), sp)
                b.record(stream)
                torch.cuda.synchronize(device)
                if it >= 2:
                    ts.append(a.elapsed_time(b) * 1e3 / 20)
            return statistics.median(ts)

        peak_gbs, _ = measured_peak()
        to_head = uly_time(0, x, y)
        to_seq = uly_time(1, y, x)
        if thd.status_read(status) != 0:
            raise RuntimeError("device status set by the Ulysses exchange")
        piece = row_bytes // cp
        # the library's rule (ulysses_tile.cu): pieces that are multiples of
        # 16 bytes below 256 B take the tile transpose, 256 B - 1 KiB take it
        # when a tile holds enough tokens, the rest go piece by piece
        tiled = cp > 1 and piece % 16 == 0
        engine = ("tile transpose (ulysses_to_heads_kernel / ulysses_to_sequence_kernel)" if tiled and piece < 256
                  else "tile transpose or row engine, by tokens per tile" if tiled and piece < 1024
                  else "row engine")
        uly = {"piece_bytes": piece, "engine": engine, "seq_to_head_us": round(to_head, 2),
               "method": "20 launches back to back per direction, per launch, median of 10",
               "head_to_seq_us": round(to_seq, 2),
               "gbs": round(swap_bytes / ((to_head + to_seq) / 2) / 1e3, 1),
               "frac_of_measured": round(swap_bytes / ((to_head + to_seq) / 2) / 1e3 / peak_gbs, 4)}

    # the pages' three passes (pack -> all-to-all -> scatter) for one z->c
    # conversion, reported against the fused swap's algorithmic bytes
    unfused = None
    if layers > 0:
        send, recv = torch.empty_like(x), torch.empty_like(x)
        ts = []
        for it in range(25):
            if it == 0 or it % 5 == 0:
                torch.cuda._sleep(200_000)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            lib.thd_pack(x.data_ptr(), send.data_ptr(), row_bytes, ctypes.byref(fwd.c), status.data_ptr(), sp)
            lib.thd_a2a_local(send.data_ptr(), recv.data_ptr(), row_bytes, ctypes.byref(fwd.c), status.data_ptr(), sp)
            lib.thd_scatter(recv.data_ptr(), y.data_ptr(), row_bytes, ctypes.byref(fwd.c), status.data_ptr(), sp)
            b.record(stream)
            torch.cuda.synchronize(device)
            if it >= 5:
                ts.append(a.elapsed_time(b) * 1e3)
        lib.thd_swap(x.data_ptr(), send.data_ptr(), row_bytes, ctypes.byref(fwd.c), status.data_ptr(), sp)
        torch.cuda.synchronize(device)
        if thd.status_read(status) != 0 or not torch.equal(send, y):
            raise RuntimeError("the three passes and the fused swap disagree")
        del send, recv
        t3 = statistics.median(ts)
        peak_gbs, _ = measured_peak()
        unfused = {"pack_a2a_scatter_us": round(t3, 2), "payload_passes": 3,
                   "gbs": round(swap_bytes / t3 / 1e3, 1),
                   "frac_of_measured": round(swap_bytes / t3 / 1e3 / peak_gbs, 4),
                   "vs_fused": "same algorithmic bytes (2 x T x row_bytes) as one fused swap"}

    # The swap in steady state: a model step does other work between swaps,
    # so a swap's input is not the previous launch's output.  Three
    # input/output buffer pairs in rotation (directions alternating): no swap
    # reads what the launch before it wrote, and the dirty lines the previous
    # launch left in L2 are written back during this one.
    steady = None
    if layers > 0:
        ins = [x] + [x.clone() for _ in range(2)]
        outs = [torch.empty_like(x) for _ in range(3)]
        routes = (fwd, bwd)
        k_box = [0]

        def rotating_swap():
            k = k_box[0]
            k_box[0] += 1
            lib.thd_swap(ins[k % 3].data_ptr(), outs[k % 3].data_ptr(), row_bytes, ctypes.byref(routes[k % 2].c),
                         status.data_ptr(), sp)

        steady_us = back_to_back_us(rotating_swap, stream, device, launches=30, reps=8, skip=2)
        if thd.status_read(status) != 0:
            raise RuntimeError("device status set by the rotating-buffer swaps")
        peak_gbs, _ = measured_peak()
        steady = {"us_per_launch": steady_us, "gbs": round(swap_bytes / steady_us / 1e3, 1),
                  "frac_of_measured": round(swap_bytes / steady_us / 1e3 / peak_gbs, 4),
                  "method": "3 input/output buffer pairs in rotation, directions alternating (no swap reads the "
                            "previous launch's output); 30 launches back to back between CUDA events, per launch, "
                            "median of 6"}
        del ins, outs

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(thd, w, x, T, cp, cu_d, row_bytes, layers, device, world, swap_bytes,
                      steps=max(12, args.steps))

    others = prep_scale = None
    if not args.no_other_configs:
        others = run_other_configs(thd, lib, w.name, device, stream, status)
        prep_scale = run_prep_at_scale(thd, lib, device, stream, status)

    peak, peak_kind = measured_peak()
    traffic = swap_traffic_record(w.name)
    result = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": n_ev,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / n_ev, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int32",
        "payload": "bf16 rows moved as raw 16-byte units",
        "data": "synthetic",
        "config": {
            "workload": w.name,
            "description": w.description,
            "cp_size": cp,
            "T": T,
            "num_docs": n_docs,
            "row_bytes": row_bytes,
            "layers": layers,
            "swaps_per_step": 2 * layers,
            "parallelism": f"{world} independent microbatch(es), one per GPU; {cp} virtual CP ranks per GPU",
            "l2": f"no flush: working set {2 * T * row_bytes / 2**30:.2f} GiB > L2 {L2_BYTES / 2**20:.0f} MiB",
        },
        "rows_per_s": round(T * 2 * layers * n_ev * world / (total_ms / 1e3), 1),
        "route_build_us": route_us,
        "swap_us_per_launch": round(swap_us, 2),
        "swap_us_distribution": swap_dist,
        "frac_of_spec_8tbs": round(achieved / SPEC_HBM_GBS, 4),
        "roofline": {
            "bound": "hbm",
            "kernel": plan_kernel_name(row_bytes),
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_kind": f"{peak_kind} copy bandwidth (read+write)",
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "algorithmic_bytes_per_launch": swap_bytes,
            "frac_dram_bytes": (round(traffic / (swap_us * 1e-6) / 1e9 / peak, 4) if traffic else None),
            "frac_steady_state": steady["frac_of_measured"] if steady else None,
        },
        "gpu_launches": launches_per_step * n_ev * world,   # every rank's, like value
        "clocks": clock_rec,
    }
    if unfused is not None:
        result["unfused"] = unfused
    if e2e is not None:
        result["e2e"] = e2e
    if prep is not None:
        result["data_prep_kernels"] = prep
    if uly is not None:
        result["ulysses_swap"] = uly
    if steady is not None:
        result["swap_steady_state"] = steady
    if others:
        result["other_configs"] = others
    if prep_scale:
        result["data_prep_at_scale"] = prep_scale
    return result, dict(x=x, T=T, cu=cu_d, w=w, row_bytes=row_bytes)


def run_other_configs(thd, lib, current, device, stream, status):
    """The second 128K workload (longtail128k: cp=8, 8 KiB rows) and the
    route-build stress workload (stress16: cp=16, 4,096 documents, 512 B
    rows), timed with the same CUDA-event method as the benchmarked
    workload: route pair and partition (single launch and back to back) and
    the swap pair (20 launches back to back, directions alternating, per
    launch).  After timing, the payload must have come back unchanged (each
    z->c swap is undone by the next c->z swap)."""
    import ctypes

    peak_gbs, peak_kind = measured_peak()
    sp = stream.cuda_stream
    out = {}
    for name in ("longtail128k", "stress16"):
        if name == current:
            continue
        w = W.BY_NAME[name]
        cu_list = W.boundaries(W.doc_lengths(name))
        T, cp, n_docs = cu_list[-1], w.cp, len(cu_list) - 1
        cu_d = torch.tensor(cu_list, dtype=torch.int32, device=device)
        x = W.payload_device(w.seed, T, w.hidden, device)
        x0 = x.clone()
        y = torch.empty_like(x)
        fwd, bwd = thd.Route.pair(T, cp, device)
        pidx = torch.empty((cp, T // cp), dtype=torch.int32, device=device)
        rb = w.row_bytes

        def pair():
            lib.thd_route_build_pair(cu_d.data_ptr(), n_docs, T, cp, ctypes.byref(fwd.c), ctypes.byref(bwd.c),
                                     status.data_ptr(), sp)

        def part():
            lib.thd_partition_indices(cu_d.data_ptr(), n_docs, T, cp, -1, pidx.data_ptr(), status.data_ptr(), sp)

        k_box = [0]

        def swap():
            k = k_box[0]
            k_box[0] += 1
            a, b, r = (x, y, fwd) if k % 2 == 0 else (y, x, bwd)
            lib.thd_swap(a.data_ptr(), b.data_ptr(), rb, ctypes.byref(r.c), status.data_ptr(), sp)

        pair()
        torch.cuda.synchronize(device)
        route = {"both_directions": single_us(pair, stream, device),
                 "both_directions_back_to_back": back_to_back_us(pair, stream, device),
                 "partition": single_us(part, stream, device),
                 "partition_back_to_back": back_to_back_us(part, stream, device)}
        swap_us = back_to_back_us(swap, stream, device, launches=20, reps=10, skip=2)   # an even count per rep
        torch.cuda.synchronize(device)
        if thd.status_read(status) != 0 or not torch.equal(x, x0):
            raise RuntimeError(f"{name}: device status set or the payload did not come back")
        swap_bytes = 2 * T * rb
        gbs = swap_bytes / swap_us / 1e3
        out[name] = {"description": w.description, "cp_size": cp, "T": T, "num_docs": n_docs, "row_bytes": rb,
                     "route_build_us": route,
                     "swap": {"kernel": plan_kernel_name(rb), "us_per_launch": swap_us, "gbs": round(gbs, 1),
                              "frac_of_measured": round(gbs / peak_gbs, 4),
                              "frac_of_spec_8tbs": round(gbs / SPEC_HBM_GBS, 4),
                              "rows_per_s": round(T / (swap_us * 1e-6), 1),
                              "algorithmic_bytes_per_launch": swap_bytes},
                     "method": "route: median single launch (GPU kept busy ahead) and 20 back to back per launch; "
                               "swap: 20 launches back to back (z->c, c->z alternating), per launch, median of 8; "
                               f"peak = {peak_kind} copy bandwidth {peak_gbs} GB/s"}
        del x, x0, y, fwd, bwd, pidx
        torch.cuda.empty_cache()
    return out


def run_e2e(thd, w, x, T, cp, cu_d, row_bytes, layers, device, world, swap_bytes, steps=12, slots=3):
    """End to end through the public API with host buffers.  Every step copies
    its input (x and the boundaries) from pinned host memory to the device,
    builds both routes, runs the layers' swap pairs and copies the result back
    to pinned host memory.  Uploads and downloads run on two copy streams of
    their own over `slots` device buffers, so uploads, downloads (the link is
    full duplex) and compute overlap.  Uploads are issued `slots - 1` steps
    ahead; before refilling a slot the host waits for the download of the
    slot's previous result (an event the download stream records).  The
    waits stay on the host because a device-side wait there would close a
    cycle of stream waits (compute on uploads, uploads on downloads,
    downloads on compute), which cost about 0.6 ms per step on GB300.  The
    timed region spans the first upload to the last download; it runs as
    many steps as the device-timed leg (at least 12), so the first upload and
    the last download, which nothing overlaps, weigh the same in both."""
    x_host = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    x_host.copy_(x)
    cu_host = cu_d.cpu().pin_memory()
    out_host = [torch.empty_like(x_host).pin_memory() for _ in range(slots)]
    xd = [torch.empty_like(x) for _ in range(slots)]
    yd = [torch.empty_like(x) for _ in range(slots)]
    cud = [torch.empty_like(cu_d) for _ in range(slots)]
    st = thd.new_status(device)
    routes = thd.Route.pair(T, cp, device)
    ks = torch.cuda.current_stream(device)
    ups, downs = torch.cuda.Stream(device), torch.cuda.Stream(device)
    cs = ups  # the link-only timings below
    ahead = slots - 1

    def run(n):
        up = [torch.cuda.Event() for _ in range(n)]
        done = [torch.cuda.Event() for _ in range(n)]
        freed = [torch.cuda.Event() for _ in range(n)]

        def upload(i):
            if i >= slots:
                freed[i - slots].synchronize()  # the slot's last result is read back
            with torch.cuda.stream(ups):
                xd[i % slots].copy_(x_host, non_blocking=True)
                cud[i % slots].copy_(cu_host, non_blocking=True)
                up[i].record(ups)

        for i in range(min(ahead, n)):
            upload(i)
        for i in range(n):
            k = i % slots
            ks.wait_event(up[i])
            fwd, bwd = thd.route_build_pair(cud[k], T, cp, status=st, routes=routes, stream=ks)
            for _ in range(layers):
                thd.swap(xd[k], fwd, out=yd[k], status=st, stream=ks)
                thd.swap(yd[k], bwd, out=xd[k], status=st, stream=ks)
            done[i].record(ks)
            with torch.cuda.stream(downs):
                downs.wait_event(done[i])
                out_host[k].copy_(xd[k], non_blocking=True)
                freed[i].record(downs)
            if i + ahead < n:
                upload(i + ahead)
        ks.wait_stream(downs)

    run(2)
    torch.cuda.synchronize(device)

    # the link alone: one pinned upload and one download of x, each timed on the copy stream
    def link_gbs(fn):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(cs):
            a.record(cs)
            fn()
            b.record(cs)
        torch.cuda.synchronize(device)
        return round(x.numel() * x.element_size() / (a.elapsed_time(b) * 1e-3) / 1e9, 1)

    h2d_gbs = link_gbs(lambda: xd[0].copy_(x_host, non_blocking=True))
    d2h_gbs = link_gbs(lambda: out_host[0].copy_(xd[0], non_blocking=True))
    barrier(world, device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(ks)
    ups.wait_stream(ks)
    downs.wait_stream(ks)
    run(steps)
    e1.record(ks)
    torch.cuda.synchronize(device)
    ms = max_over_ranks(e0.elapsed_time(e1), world, device)
    ref = x.cpu()
    if thd.status_read(st) != 0 or not all(torch.equal(o, ref) for o in out_host):
        raise RuntimeError("e2e pass produced a wrong result")
    bytes_all = sum_over_ranks(float(swap_bytes * 2 * layers * steps), world, device)
    return {"value": round(bytes_all / (ms / 1e3) / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": int(x.numel() * x.element_size() + cu_d.numel() * 4),
            "d2h_bytes_per_step": int(x.numel() * x.element_size()),
            "ms_per_step": round(ms / steps, 3), "steps": steps,
            "overlap": f"uploads ({ahead} steps ahead) and downloads on two copy streams, {slots} buffer slots, "
                       "against compute; slot reuse waits on the host",
            "link_gbs": {"h2d": h2d_gbs, "d2h": d2h_gbs}}


def run_prep_at_scale(thd, lib, device, stream, status, B=64, S=262144, cp=8, depth=3):
    """The data-preparation kernels on 64 raw rows of 262,144 tokens (16.8 M,
    drawn like the pipeline workload's rows), where launch latency no longer
    hides them: packing, labels with three MTP depths in both layouts, and
    the partition of every rank.  Each: launches back to back between CUDA
    events, per launch, median; bytes per launch are the algorithmic ones
    (packing: raw tokens read + packed tokens and boundaries written; labels:
    tokens read + (depth + 1) x (4 + 1) bytes + 1 valid byte written per
    position; partition: 4 bytes written per position)."""
    import ctypes

    peak_gbs, peak_kind = measured_peak()
    sp = stream.cuda_stream
    raw = torch.from_numpy(W.raw_pipeline_tokens(W.SEED + 4, B=B, S=S)).to(device)
    tok, cu_v, cu = thd.pack_docs(raw, W.EOD_ID, 2 * cp, pad_id=0)
    T, n = tok.numel(), cu.numel() - 1
    cap_tok, cap_docs = B * S * 2 * cp, B * S + 1
    ptok = torch.empty(cap_tok, dtype=torch.int32, device=device)
    pcu_v = torch.empty(cap_docs, dtype=torch.int32, device=device)
    pcu = torch.empty(cap_docs, dtype=torch.int32, device=device)
    counts = torch.zeros(2, dtype=torch.int64, device=device)
    ws = torch.empty(lib.thd_pack_docs_workspace_bytes(B, S), dtype=torch.uint8, device=device)
    labels = torch.empty((depth + 1, T), dtype=torch.int32, device=device)
    lmask = torch.empty((depth + 1, T), dtype=torch.uint8, device=device)
    valid = torch.empty((T,), dtype=torch.uint8, device=device)
    pidx = torch.empty((cp, T // cp), dtype=torch.int32, device=device)
    calls = {
        "pack_docs": (lambda: lib.thd_pack_docs(raw.data_ptr(), B, S, W.EOD_ID, 0, 0, 2 * cp, 0, None, ptok.data_ptr(),
                                                cap_tok, pcu_v.data_ptr(), pcu.data_ptr(), None, None, cap_docs,
                                                counts.data_ptr(), ws.data_ptr(), ws.numel(), status.data_ptr(), sp),
                      4 * B * S + 4 * T + 8 * (n + 1)),
        "roll_labels": (lambda: lib.thd_roll_labels(tok.data_ptr(), cu_v.data_ptr(), cu.data_ptr(), n, T, depth, 0, None,
                                                    None, labels.data_ptr(), lmask.data_ptr(), valid.data_ptr(),
                                                    status.data_ptr(), sp),
                        4 * T + (depth + 1) * 5 * T + T),
        "roll_labels_zigzag": (lambda: lib.thd_roll_labels_zigzag(tok.data_ptr(), cu_v.data_ptr(), cu.data_ptr(), n, T,
                                                                  cp, depth, 0, None, None, labels.data_ptr(),
                                                                  lmask.data_ptr(), valid.data_ptr(), status.data_ptr(),
                                                                  sp),
                               4 * T + (depth + 1) * 5 * T + T),
        "partition": (lambda: lib.thd_partition_indices(cu.data_ptr(), n, T, cp, -1, pidx.data_ptr(), status.data_ptr(),
                                                        sp),
                      4 * T),
    }
    out = {"raw_rows": [B, S], "T": T, "num_docs": n, "cp_size": cp, "mtp_depth": depth,
           "method": "3 launches back to back between CUDA events, per launch, median of 6; peak = "
                     f"{peak_kind} copy bandwidth {peak_gbs} GB/s"}
    for name, (fn, nbytes) in calls.items():
        us = back_to_back_us(fn, stream, device, launches=3, reps=8, skip=2)
        out[name] = {"us": us, "algorithmic_bytes": int(nbytes), "gbs": round(nbytes / us / 1e3, 1),
                     "frac_of_measured": round(nbytes / us / 1e3 / peak_gbs, 4)}
    torch.cuda.synchronize(device)
    if thd.status_read(status) != 0:
        raise RuntimeError("device status set by the data-preparation kernels at scale")
    del raw, ptok, labels, lmask, valid, pidx, ws
    torch.cuda.empty_cache()
    return out


def run_cp_exchange(args, rank, world, local):
    """The conversion between GPUs: every rank is one CP rank holding its own
    shard.  A step builds both routes on every GPU (no host synchronisation),
    reads this rank's split sizes and identity flags to the host once per
    direction (the collective needs them there), then runs every layer's
    z->c and c->z exchange (per-rank pack kernel, NCCL all_to_all_single,
    per-rank scatter kernel).  value = payload bytes of the whole batch per
    conversion (2 x T x row_bytes, read + write), summed over conversions,
    per second of the slowest rank's step time."""
    import context_packed_sequence_gb300 as thd

    w = W.BY_NAME[args.workload]
    if w.name == "pipeline" or w.cp != world:
        raise SystemExit(f"--cp-exchange needs --gpus equal to the workload's cp ({w.name}: cp={w.cp}, "
                         f"world={world}) and a workload with fixed boundaries")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    layers = args.layers if args.layers is not None else 48
    cu_list = W.boundaries(W.doc_lengths(w.name))
    T, cp = cu_list[-1], w.cp
    S = T // cp
    cu_d = torch.tensor(cu_list, dtype=torch.int32, device=device)
    shard = W.payload_device(w.seed, T, w.hidden, device)[rank * S:(rank + 1) * S].clone()   # zigzag shard
    status = thd.new_status(device)
    routes = thd.Route.pair(T, cp, device)

    launches = [0]

    def step():
        fwd, bwd = thd.route_build_pair(cu_d, T, cp, status=status, routes=routes)
        ex_f, ex_b = thd.CpExchange.from_route(fwd, rank), thd.CpExchange.from_route(bwd, rank)
        # libthd kernels per step: the route build, then pack and scatter of
        # every exchange unless that side is the identity (zero-copy)
        launches[0] = 1 + layers * sum(2 - e.send_identity - e.recv_identity for e in (ex_f, ex_b))
        a = shard
        for _ in range(layers):
            a = ex_b(ex_f(a))
        return a

    for _ in range(args.warmup):
        back = step()
    torch.cuda.synchronize(device)
    if not torch.equal(back, shard):
        raise RuntimeError("the exchanges there and back did not return the shard")
    stream = torch.cuda.current_stream(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world, device)
    torch.cuda.synchronize(device)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(device)
    barrier(world, device)
    ms = max_over_ranks(e0.elapsed_time(e1), world, device)
    conv_bytes = 2 * T * w.row_bytes
    value = conv_bytes * 2 * layers * args.steps / (ms / 1e3) / 1e9
    return {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4), "higher_is_better": True,
        "scaling": "strong", "vs_baseline": None, "dtype": "int32", "data": "synthetic", "mode": "cp_exchange",
        "config": {"workload": w.name, "cp_size": cp, "T": T, "row_bytes": w.row_bytes, "layers": layers,
                   "parallelism": f"cp{cp}: one CP rank per GPU, per-rank pack/scatter kernels around an NCCL "
                                  "all_to_all_single; split sizes read to the host once per direction per step"},
        "gpu_launches": int(sum_over_ranks(float(launches[0] * args.steps), world, device)),
    }


# ---------------------------------------------------------------------------
# the CPU oracle (cpu_baseline leg and --impl reference)
# ---------------------------------------------------------------------------

def oracle_payload(w, T):
    """The workload's payload as host bytes [T, row_bytes] (drawn on the host)."""
    x = W.payload_host(w.seed, T, w.hidden)
    return x.contiguous().view(torch.uint8).reshape(T, -1).numpy()


def oracle_cu(w):
    if w.name == "pipeline":
        import oracle
        raw = W.raw_pipeline_tokens(w.seed)
        _, _, cu = oracle.pack_docs(raw.tolist(), W.EOD_ID, 2 * w.cp, pad_id=0)
        return cu
    return W.boundaries(W.doc_lengths(w.name))


def oracle_step(cu, T, cp, direction, xb):
    """One bounded sample: the oracle builds one direction's route token by
    token and applies it (pack -> all-to-all -> scatter) to the full payload."""
    import oracle
    rt = oracle.build_route(cu, T, cp, direction)
    _, _, out = oracle.apply_route(xb, rt)
    return out


def run_cpu_baseline(w, budget_s):
    cu = oracle_cu(w)
    T = cu[-1]
    xb = oracle_payload(w, T)
    swap_bytes = 2 * T * w.row_bytes
    done, t0 = 0, time.perf_counter()
    while True:
        oracle_step(cu, T, w.cp, done % 2, xb)
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return {"value": round(done * swap_bytes / el / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "host_cpus": os.cpu_count(),
            "sample": f"{done} oracle swap(s) of the full {w.name} workload (T={T}, {w.row_bytes} B rows), "
                      f"each = per-token route build of one direction + pack/all-to-all/scatter row by row, "
                      f"pure Python on 1 thread, {el:.1f} s"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    w = W.BY_NAME[args.workload]
    cu = oracle_cu(w)
    T = cu[-1]
    xb = oracle_payload(w, T)
    swap_bytes = 2 * T * w.row_bytes
    for i in range(args.warmup):
        oracle_step(cu, T, w.cp, i % 2, xb)
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle_step(cu, T, w.cp, i % 2, xb)
    el = time.perf_counter() - t0
    value = args.steps * swap_bytes / el / 1e9
    sample = (f"each step = one oracle swap of the full {w.name} workload (T={T}, {w.row_bytes} B rows): "
              f"per-token route build of one direction + pack/all-to-all/scatter row by row, 1 thread")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(el * 1e3 / max(args.steps, 1), 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int32",
        "data": "synthetic",
        "config": {"workload": w.name, "description": w.description, "cp_size": w.cp, "T": T,
                   "row_bytes": w.row_bytes},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "host_cpus": os.cpu_count(), "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    rank, world, local = setup_dist(args)
    try:
        if args.impl == "reference":
            res = run_reference(args, rank, world)
            if res is not None:
                print(json.dumps(res), flush=True)
            return
        if not torch.cuda.is_available():
            raise SystemExit("bench.py: the thd arm needs a CUDA GPU")
        if args.only_prep_at_scale:
            import context_packed_sequence_gb300 as thd
            from context_packed_sequence_gb300 import _lib as L
            device = torch.device("cuda", local)
            torch.cuda.set_device(device)
            clocks = ClockSampler(smi_gpu_id(device)).start()
            prep = run_prep_at_scale(thd, L.load(), device, torch.cuda.current_stream(device), thd.new_status(device))
            res = {"data_prep_at_scale": prep, "clocks": clocks.stop()}
            if rank == 0:
                print(json.dumps(res), flush=True)
            return
        if args.cp_exchange:
            res = run_cp_exchange(args, rank, world, local)
            if rank == 0:
                print(json.dumps(res), flush=True)
            return
        res, _ = run_thd(args, rank, world, local)
        if rank == 0:
            if not args.no_cpu_baseline and world == 1:
                res["cpu_baseline"] = run_cpu_baseline(W.BY_NAME[args.workload], args.cpu_budget)
            print(json.dumps(res), flush=True)
    finally:
        if world > 1 and dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
