#!/usr/bin/env python3
"""Benchmark of the multi-scale deformable attention core on B300 (libmsda).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one pass of the hot path over one batch of synthetic input: by default the
forward of the encoder-shaped workload (B=2, 4-level pyramid 100x150..13x19, Nq=Nin=19947,
M=8, D=32, P=4, fp32), i.e. the coordinate transform, corner gather, interpolation /
weighted sum and store.  Other workloads: tiny2d, decoder2d, volume3d (forward) and
encoder2d_bwd (zero-fill + backward).

Prints ONE JSON line (rank 0).  `value` is samples (B*Nq*M*L*P) per second over all ranks,
timed on the device with CUDA events on the launching stream over exactly K steps
(barrier + synchronize on both sides, max over ranks); the K steps are captured into one
CUDA graph so that host call overhead does not hide kernel time.  L2 is kept cold by rotating over
input sets whose total size is more than twice the L2 capacity.  `e2e` is the same metric
through the public binding with pinned host buffers, host->device copies of the inputs and
the device->host copy of the output inside the timed region (steps pipelined on three
streams, as a caller streaming batches would).  `cpu_baseline` times the CPU
oracle (test infrastructure) on the host, single-threaded.

Under torchrun (N > 1) every rank runs its own batch of the workload (weak scaling; no
collective on the data path; NCCL is used only for the barrier and the max of the times).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "sampled points/s (B·Nq·M·L·P per s) and achieved HBM GB/s vs ~8 TB/s peak"
UNIT = "samples/s"
NOMINAL_HBM_GBS = 7700.0  # B300 HBM3e nominal bandwidth
FALLBACK_HBM_GBS = 6400.0
L1_WAVEFRONT_BYTES = 128   # bytes one L1 data-pipe wavefront delivers; one per SM clock
# Rate of the L2 reduction units in 32-byte sector updates per second: the reduce_l2 probe
# (`bench.py --probe reduce_l2`: red.global.add.v4.f32 of random 128-byte rows, 8 lanes
# per row, four whole sectors per request) measured 49.6 G rows/s on a B300.
L2_RED_SECTORS_PER_S = 4 * 49.6e9
PROFILE_DIR = os.path.join(ROOT, "profiles")
KERNEL_SRC_DIR = os.path.join(ROOT, "scale_deformable_attention_msda3d_b300", "csrc")


# ----------------------------------------------------------------------------- helpers


# Sources that decide what the forward / backward kernels do (shared headers and the ABI
# layer that packs their parameters, plus the kernel file itself).
KERNEL_FILES = {
    "forward": ("common.cuh", "msda_internal.h", "msda_abi.cpp", "msda_forward.cuh",
                "msda_forward.cu", "msda_forward_f32_2d.cu", "msda_forward_f32_3d.cu",
                "msda_forward_bf16_2d.cu", "msda_forward_bf16_3d.cu", "msda_forward_rt_f32_2d.cu",
                "msda_forward_rt_f32_3d.cu", "msda_forward_rt_bf16_2d.cu",
                "msda_forward_rt_bf16_3d.cu"),
    "backward": ("common.cuh", "msda_internal.h", "msda_abi.cpp", "msda_backward.cuh",
                 "msda_backward.cu", "msda_backward_2d.cu", "msda_backward_3d.cu",
                 "msda_backward_fused_2d.cu", "msda_backward_fused_3d.cu"),
}


def _code_only(text: str) -> str:
    """C / C++ / CUDA source with comments and whitespace removed (string literals with
    comment markers are not expected in these sources)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return re.sub(r"\s+", "", text)


def kernel_source_hash(kind: str = "forward") -> str:
    """sha256 over the code (comments and whitespace stripped) of one kernel family of
    libmsda: it identifies the measured kernels, and a profile taken on other code no longer
    describes them."""
    h = hashlib.sha256()
    for f in KERNEL_FILES[kind]:
        h.update(f.encode())
        h.update(_code_only(open(os.path.join(KERNEL_SRC_DIR, f)).read()).encode())
    return h.hexdigest()


def recorded_counter(workload: str, mode: str = "", key: str = "dram_bytes_per_launch"):
    """A per-launch counter of the dominant kernel (`key`: dram_bytes_per_launch or
    l1_wavefronts_per_launch) from a committed ncu summary, if that summary was taken on
    the current sources of the kernel family (else None).  A summary names its bench
    workload, with "+order" / "+fused" / "+prune<t>" / "+order_once" appended for those
    modes."""
    src = kernel_source_hash("backward" if workloads.WORKLOADS[workload].backward else "forward")
    want = workload + mode
    if not os.path.isdir(PROFILE_DIR):
        return None
    for f in sorted(os.listdir(PROFILE_DIR)):
        if not f.endswith((".md", ".txt")):
            continue
        text = open(os.path.join(PROFILE_DIR, f)).read()
        m_w = re.search(r"^bench_workload:\s*(\S+)", text, re.M)
        m_h = re.search(r"^kernel_source_sha256:\s*([0-9a-f]{64})", text, re.M)
        m_t = re.search(r"^" + re.escape(key) + r":\s*([0-9.eE+]+)", text, re.M)
        if m_w and m_h and m_t and m_w.group(1) == want and m_h.group(1) == src:
            return float(m_t.group(1))
    return None


def recorded_traffic(workload: str, mode: str = ""):
    """DRAM bytes per launch from a committed ncu summary of the current sources."""
    return recorded_counter(workload, mode, "dram_bytes_per_launch")


def l1_ceiling(w, corner_rows: int, wavefronts, sm_count: int, sm_mhz, launch_s: float,
               alg_bytes: int, hbm_peak_gbs: float) -> dict:
    """The SM-side ceiling of the gather: every in-level corner row of every sample passes
    through an SM's L1 data pipe into registers, which delivers one 128-byte wavefront per
    SM clock.  rows_floor_us is the time those rows alone need on all SMs at the sampled
    clock (the minimum of any design that brings each corner row on chip once); floor_us
    the time of the wavefronts the dominant kernel issued per launch (corner rows plus its
    tap exchange, loads of locations and weights and stores), from the committed ncu
    summary of the same sources; frac = that floor over the measured launch time.
    hbm_frac_ceiling is the HBM-roofline fraction a launch at rows_floor_us would reach."""
    esize = 2 if w.dtype == "bf16" else 4
    per_row = max(1, -(-(w.D * esize) // L1_WAVEFRONT_BYTES))
    rows_wf = corner_rows * per_row
    if not sm_mhz:
        return {"bound": "l1_data_pipe", "corner_rows_per_launch": corner_rows, "frac": None}
    cyc_us = sm_count * float(sm_mhz)                      # wavefronts per microsecond
    rows_floor = rows_wf / cyc_us
    floor = wavefronts / cyc_us if wavefronts else None
    launch_us = launch_s * 1e6
    return {"bound": "l1_data_pipe", "unit": "wavefronts (128 B; one per SM clock)",
            "corner_rows_per_launch": corner_rows, "rows_wavefronts_per_launch": rows_wf,
            "rows_floor_us": rows_floor, "rows_frac": rows_floor / launch_us,
            "wavefronts_per_launch": wavefronts, "floor_us": floor,
            "frac": (floor / launch_us) if floor else None,
            "sm_count": sm_count, "sm_mhz": float(sm_mhz),
            "hbm_frac_ceiling": alg_bytes / (rows_floor * 1e-6) / 1e9 / hbm_peak_gbs,
            "source": "rows counted on the host from the inputs; wavefronts from the ncu "
                      "summary of the current kernel sources (null when none matches)"}


def l2_reduction_ceiling(w, corner_rows: int, launch_s: float) -> dict:
    """The L2-side ceiling of the backward: every in-level corner row of every sample adds
    its weighted grad_out into one D-channel fp32 row of grad_value with vector reductions
    issued in runs of whole 32-byte sectors, D * 4 / 32 sector updates per row.  floor_us is
    the time those updates need at the rate the reduce_l2 probe measured
    (L2_RED_SECTORS_PER_S); frac = that floor over the measured launch time."""
    sectors = corner_rows * max(1, -(-(w.D * 4) // 32))
    floor_us = sectors / L2_RED_SECTORS_PER_S * 1e6
    return {"bound": "l2_reductions", "unit": "32-byte sector updates",
            "sector_updates_per_launch": sectors, "rate_per_s": L2_RED_SECTORS_PER_S,
            "floor_us": floor_us, "frac": floor_us / (launch_s * 1e6),
            "source": "rows counted on the host from the inputs; the rate measured by the "
                      "reduce_l2 probe on a B300 (49.6 G 128-byte rows/s)"}


def l2_bytes(dev) -> int:
    """L2 capacity of the device (bytes), as the driver reports it."""
    import torch
    return int(torch.cuda.get_device_properties(dev).L2_cache_size)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            return float(d["hbm_gbs"]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def unique_value_rows(w: workloads.Workload, inp) -> int:
    """Distinct (batch, value row, head) rows touched by at least one corner that lies
    inside its level: the value bytes a perfect cache would read once."""
    return value_row_counts(w, inp)[0]


def value_row_counts(w: workloads.Workload, inp):
    """(distinct rows, all in-level corner rows) of one pass: every in-level corner of
    every sample brings one D-channel value row of one head on chip."""
    loc = inp["sampling_locations"].astype(np.float64)
    B, Nq, M, L, P, nd = loc.shape
    starts = inp["level_start_index"]
    ids = []
    b_idx = np.arange(B).reshape(B, 1, 1, 1)
    m_idx = np.arange(M).reshape(1, 1, M, 1)
    for l in range(L):
        shape = [int(s) for s in inp["spatial_shapes"][l]]
        ext = shape[::-1]                                   # (W, H[, Z])
        pix = loc[:, :, :, l] * np.array(ext, dtype=np.float64) - 0.5   # [B,Nq,M,P,nd]
        ok_s = np.all((pix > -1) & (pix < np.array(ext)), axis=-1)
        i0 = np.floor(np.where(np.isfinite(pix), pix, -5)).astype(np.int64)
        for c in range(2 ** nd):
            d = np.array([(c >> k) & 1 for k in range(nd)])
            idx = i0 + d
            inside = ok_s & np.all((idx >= 0) & (idx < np.array(ext)), axis=-1)
            if nd == 2:
                row = idx[..., 1] * ext[0] + idx[..., 0]
            else:
                row = (idx[..., 2] * ext[1] + idx[..., 1]) * ext[0] + idx[..., 0]
            gid = ((b_idx * w.Nin + starts[l] + row) * M + m_idx)
            ids.append(gid[inside])
    allrows = np.concatenate(ids)
    return int(np.unique(allrows).size), int(allrows.size)


def algorithmic_bytes(w: workloads.Workload, inp, counts=None) -> dict:
    """Algorithmic bytes of one pass; `counts` = value_row_counts(w, inp) if known."""
    esize = 2 if w.dtype == "bf16" else 4
    row = w.D * esize
    uniq = (counts or value_row_counts(w, inp))[0] * row
    loc_b = inp["sampling_locations"].nbytes
    attn_b = inp["attention_weights"].nbytes
    out_b = w.B * w.Nq * w.M * w.D * esize
    whole_value = w.B * w.Nin * w.M * row
    if not w.backward:
        total = uniq + loc_b + attn_b + out_b
        parts = dict(unique_value=uniq, locations=loc_b, weights=attn_b, out=out_b)
    else:
        gv = w.B * w.Nin * w.M * w.D * 4
        total = uniq + loc_b + attn_b + out_b + gv + loc_b + attn_b + gv   # + zero-fill
        parts = dict(unique_value=uniq, locations=loc_b, weights=attn_b, grad_out=out_b,
                     grad_value=gv, grad_locations=loc_b, grad_weights=attn_b,
                     grad_value_zero_fill=gv)
    parts["whole_value_tensor"] = whole_value
    return dict(total=int(total), parts=parts)


class ClockSampler:
    """Samples SM clock and clock-event (throttle) reasons while the GPU works: through
    NVML when pynvml imports, else by running nvidia-smi in loop mode."""

    REASONS = {
        "gpu_idle": 0x1, "applications_clocks_setting": 0x2, "sw_power_cap": 0x4,
        "hw_slowdown": 0x8, "sync_boost": 0x10, "sw_thermal_slowdown": 0x20,
        "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80,
        "display_clock_setting": 0x100,
    }

    def __init__(self, device_index: int, pci_bus_id: str = None, period_s: float = 0.005):
        self.samples = []
        self.reasons = set()
        self.max_mhz = None
        self.period = period_s
        self.source = None
        self.error = None
        self._stop = threading.Event()
        self._t = None
        self._proc = None
        self._smi_id = pci_bus_id or str(device_index)
        try:
            import pynvml
            pynvml.nvmlInit()
            self._nvml = pynvml
            self._h = (pynvml.nvmlDeviceGetHandleByPciBusId(pci_bus_id) if pci_bus_id
                       else pynvml.nvmlDeviceGetHandleByIndex(device_index))
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self._h, pynvml.NVML_CLOCK_SM)
            self.source = "nvml"
        except Exception as e:
            self._nvml = None
            self.error = f"pynvml: {e}"
            import shutil
            if shutil.which("nvidia-smi"):
                self.source = "nvidia-smi"

    def _add(self, mhz, max_mhz, mask):
        self.samples.append(float(mhz))
        if max_mhz:
            self.max_mhz = float(max_mhz)
        for name, bit in self.REASONS.items():
            if mask & bit:
                self.reasons.add(name)

    def sample_once(self):
        if self._nvml is None:
            return
        n = self._nvml
        try:
            self._add(n.nvmlDeviceGetClockInfo(self._h, n.NVML_CLOCK_SM), None,
                      n.nvmlDeviceGetCurrentClocksEventReasons(self._h))
        except Exception:
            pass

    def _run_nvml(self):
        while not self._stop.is_set():
            self.sample_once()
            time.sleep(self.period)

    def _run_smi(self):
        for line in self._proc.stdout:
            parts = [t.strip() for t in line.split(",")]
            if len(parts) != 3:
                continue
            try:
                self._add(float(parts[0]), float(parts[1]), int(parts[2], 16))
            except ValueError:
                continue

    def __enter__(self):
        if self.source == "nvml":
            self._t = threading.Thread(target=self._run_nvml, daemon=True)
            self._t.start()
        elif self.source == "nvidia-smi":
            import subprocess
            self._proc = subprocess.Popen(
                ["nvidia-smi", "-i", self._smi_id,
                 "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._run_smi, daemon=True)
            self._t.start()
            time.sleep(0.3)          # let the first samples arrive before the timed work
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self._proc is not None:
            time.sleep(0.05)
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except Exception:
                self._proc.kill()
        if self._t is not None:
            self._t.join(timeout=5)

    def summary(self):
        if self.source is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "error": self.error}
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "samples": len(self.samples),
                "reasons": sorted(self.reasons - {"gpu_idle"}), "source": self.source}


def pci_bus_id(dev) -> str:
    """nvidia-smi / NVML style bus id of a torch CUDA device (None if unknown)."""
    try:
        import torch
        p = torch.cuda.get_device_properties(dev)
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except Exception:
        return None


# ----------------------------------------------------------------------------- distributed


def dist_setup(want_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    elif want_gpus > 1:
        print(f"--gpus {want_gpus} needs torchrun (one process per GPU); running 1 rank",
              file=sys.stderr)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _reduce(x: float, world: int, op: str) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def all_max(x: float, world: int) -> float:
    return _reduce(x, world, "max")


def all_sum(x: float, world: int) -> float:
    return _reduce(x, world, "sum")


def aggregate(t_rank_s: float, samples_rank: int, steps: int, world: int):
    """Whole-job throughput: samples of all ranks over the slowest rank's time."""
    t_max = all_max(t_rank_s, world)
    samples_all = all_sum(float(samples_rank), world) * steps
    return samples_all / t_max, t_max


# ----------------------------------------------------------------------------- our arm


def to_device(inp, w, dev):
    import torch
    if w.dtype == "bf16":
        value = torch.from_numpy(inp["value_bits"].view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        value = torch.from_numpy(inp["value"]).to(dev)
    d = dict(value=value,
             loc=torch.from_numpy(inp["sampling_locations"]).to(dev),
             attn=torch.from_numpy(inp["attention_weights"]).to(dev))
    if w.backward:
        if w.dtype == "bf16":
            d["grad_out"] = torch.from_numpy(inp["grad_out_bits"].view(np.int16)).to(dev).view(
                torch.bfloat16)
        else:
            d["grad_out"] = torch.from_numpy(inp["grad_out"]).to(dev)
    return d


def fused_byte_inputs(w, f):
    """Sampling locations of fused inputs (reference + offset / extent in fp32, as the
    kernel forms them) for counting the unique value rows; host-side bookkeeping only."""
    ext = f["spatial_shapes"][:, ::-1].astype(np.float32)
    loc = (f["reference_points"][:, :, None, :, None, :]
           + f["sampling_offsets"] / ext[None, None, None, :, None, :])
    return dict(sampling_locations=loc, spatial_shapes=f["spatial_shapes"],
                level_start_index=f["level_start_index"],
                attention_weights=f["attention_logits"])


def make_step(msda, w, inp, bufs, stream, ordered=None, prune=0.0, fused=False):
    """Returns step(i): one pass of the hot path on input set i % len(bufs).  With
    ordered = "step", each step first computes the locality-aware query order of its input
    set (msda_query_order) and then runs the ordered forward, both inside the step; with
    "once", the order of every input set is computed here, before any timing, and the step
    runs only the ordered forward.  With `prune` > 0 it runs the pruned forward (samples
    with |A| < prune skipped)."""
    shapes, starts = inp["spatial_shapes"], inp["level_start_index"]
    if ordered and w.backward:
        # the ordered backward; the order as for the forward (once per input set, or in
        # each step)
        fn = msda.msda2d_backward_ordered if w.ndim == 2 else msda.msda3d_backward_ordered
        if ordered == "once":
            with __import__("torch").cuda.stream(stream):
                for b in bufs:
                    msda.msda_query_order(b["loc"], query_order=b["order"], workspace=b["ws"],
                                          stream=stream)

        def step(i):
            b = bufs[i % len(bufs)]
            if ordered != "once":
                msda.msda_query_order(b["loc"], query_order=b["order"], workspace=b["ws"],
                                      stream=stream)
            fn(b["value"], shapes, starts, b["loc"], b["attn"], b["order"], b["grad_out"],
               grad_value=b["gv"], grad_sampling_locations=b["gl"],
               grad_attention_weights=b["ga"], stream=stream)
        # zero-fill and backward (+ keys, scan, scatter of the order in each step)
        return step, 2 if ordered == "once" else 5
    if fused and w.backward:
        fn = msda.msda2d_backward_fused if w.ndim == 2 else msda.msda3d_backward_fused

        def step(i):
            b = bufs[i % len(bufs)]
            fn(b["value"], shapes, starts, b["ref"], b["loc"], b["attn"], b["grad_out"],
               stream=stream, grad_value=b["gv"], grad_sampling_offsets=b["gl"],
               grad_attention_logits=b["ga"], grad_reference_points=b["gref"])
        # zero-fill, backward, reference-point epilogue (+ the logit epilogue when the
        # generic kernels run, i.e. (L, P) outside the compiled pairs)
        tiled = w.P == 4 and w.L in (1, 4)
        return step, 3 if tiled else 4
    if fused:
        fn = msda.msda2d_forward_fused if w.ndim == 2 else msda.msda3d_forward_fused

        def step(i):
            b = bufs[i % len(bufs)]
            fn(b["value"], shapes, starts, b["ref"], b["loc"], b["attn"], out=b["out"],
               stream=stream)
        return step, 1
    if prune > 0:
        fn = msda.msda2d_forward_pruned if w.ndim == 2 else msda.msda3d_forward_pruned

        def step(i):
            b = bufs[i % len(bufs)]
            fn(b["value"], shapes, starts, b["loc"], b["attn"], prune, out=b["out"],
               stream=stream)
        return step, 1
    if ordered == "once":
        fn = msda.msda2d_forward_ordered if w.ndim == 2 else msda.msda3d_forward_ordered
        with __import__("torch").cuda.stream(stream):
            for b in bufs:
                msda.msda_query_order(b["loc"], query_order=b["order"], workspace=b["ws"],
                                      stream=stream)

        def step(i):
            b = bufs[i % len(bufs)]
            fn(b["value"], shapes, starts, b["loc"], b["attn"], b["order"], out=b["out"],
               stream=stream)
        return step, 1
    if ordered:
        fn = msda.msda2d_forward_ordered if w.ndim == 2 else msda.msda3d_forward_ordered

        def step(i):
            b = bufs[i % len(bufs)]
            msda.msda_query_order(b["loc"], query_order=b["order"], workspace=b["ws"],
                                  stream=stream)
            fn(b["value"], shapes, starts, b["loc"], b["attn"], b["order"], out=b["out"],
               stream=stream)
        return step, 4          # keys, scan, scatter, forward (plus a histogram memset)
    if not w.backward:
        fn = msda.msda2d_forward if w.ndim == 2 else msda.msda3d_forward

        def step(i):
            b = bufs[i % len(bufs)]
            fn(b["value"], shapes, starts, b["loc"], b["attn"], out=b["out"], stream=stream)
        return step, 1
    fn = msda.msda2d_backward if w.ndim == 2 else msda.msda3d_backward

    def step(i):
        b = bufs[i % len(bufs)]
        fn(b["value"], shapes, starts, b["loc"], b["attn"], b["grad_out"],
           grad_value=b["gv"], grad_sampling_locations=b["gl"],
           grad_attention_weights=b["ga"], stream=stream)
    return step, 2


def cpu_baseline(w, inp, budget_s: float = 10.0, fused: bool = False):
    """The oracle as it stands (C, double precision) on the full workload, repeated until
    about budget_s of wall time; samples per second.  The forward is timed on one host
    thread and on all of them (the oracle's forward split into blocks of queries, one
    OpenMP thread each; every output computed as in the serial call); the backward, whose
    grad_value sums are serial, on one thread.  `fused`: the oracle's fused forward /
    backward on reference points, offsets and logits."""
    import oracle
    oracle.build()
    args = [np.ascontiguousarray(inp[k], dtype=np.float64) for k in
            ("value", "sampling_locations", "attention_weights")]
    shapes, starts = inp["spatial_shapes"], inp["level_start_index"]
    g = np.ascontiguousarray(inp["grad_out"], dtype=np.float64) if w.backward else None

    def one(threads):
        if fused:
            pro = (inp["reference_points"], inp["sampling_offsets"], inp["attention_logits"])
            if w.backward:
                oracle.backward_fused(w.ndim, args[0], shapes, starts, *pro, g)
            else:
                oracle.forward_fused(w.ndim, args[0], shapes, starts, *pro, threads=threads)
        elif w.backward:
            oracle.backward(w.ndim, args[0], shapes, starts, args[1], args[2], g)
        else:
            oracle.forward(w.ndim, args[0], shapes, starts, args[1], args[2], threads=threads)

    def timed(threads, budget):
        runs, t0 = 0, time.perf_counter()
        while True:
            one(threads)
            runs += 1
            el = time.perf_counter() - t0
            if el >= budget:
                return runs, el

    what = f"the {w.name} workload ({w.samples} samples each)"
    if w.backward:
        runs, el = timed(1, budget_s)
        return {"value": w.samples * runs / el, "unit": UNIT, "cores": 1, "kind": "oracle",
                "sample": f"{runs} full pass(es) of {what}, {el:.1f} s, 1 thread (the "
                          "backward's grad_value sums are serial), fp64"}
    n_all = oracle.default_threads()
    r1, e1 = timed(1, budget_s / 2)
    rn, en = timed(0, budget_s / 2)
    return {"value": w.samples * rn / en, "unit": UNIT, "cores": n_all, "kind": "oracle",
            "sample": f"{rn} full pass(es) of {what}, {en:.1f} s, {n_all} threads (OpenMP "
                      "over blocks of 64 queries), fp64",
            "single_core": {"value": w.samples * r1 / e1, "unit": UNIT, "cores": 1,
                            "sample": f"{r1} full pass(es), {e1:.1f} s, 1 thread"},
            "host_cpus": os.cpu_count()}


def run_ours(args):
    import torch
    import scale_deformable_attention_msda3d_b300 as msda

    rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    msda.load()
    w = workloads.WORKLOADS[args.workload]
    if args.fused:
        # loc / attn slots carry the offsets and logits; ref the reference points
        f = workloads.make_fused_inputs(w, seed=w.seed + rank)
        inp = dict(f, sampling_locations=f["sampling_offsets"],
                   attention_weights=f["attention_logits"])
        if w.backward:  # the backward workload's upstream gradient
            full = workloads.make_inputs(w, seed=w.seed + rank)
            inp.update({k: full[k] for k in ("grad_out", "grad_out_bits") if k in full})
    else:
        inp = workloads.make_inputs(w, seed=w.seed + rank)
    base = to_device(inp, w, dev)
    if args.fused:
        base["ref"] = torch.from_numpy(inp["reference_points"]).to(dev)
    esize = 2 if w.dtype == "bf16" else 4
    set_bytes = sum(t.numel() * t.element_size() for t in base.values())
    set_bytes += w.B * w.Nq * w.M * w.D * esize
    if w.backward:
        set_bytes += base["value"].numel() * 4 + base["loc"].numel() * 4 + base["attn"].numel() * 4
    l2 = l2_bytes(dev)
    n_sets = max(2, int(np.ceil(2 * l2 / set_bytes)) + 1)
    bufs = []
    for i in range(n_sets):
        b = {k: (v if i == 0 else v.clone()) for k, v in base.items()}
        b["out"] = torch.empty((w.B, w.Nq, w.M * w.D), dtype=b["value"].dtype, device=dev)
        if w.backward:
            b["gv"] = torch.empty(b["value"].shape, dtype=torch.float32, device=dev)
            b["gl"] = torch.empty_like(b["loc"])
            b["ga"] = torch.empty_like(b["attn"])
            if args.fused:
                b["gref"] = torch.empty_like(b["ref"])
        if args.order:
            b["order"] = torch.empty((w.B, w.Nq), dtype=torch.int32, device=dev)
            b["ws"] = torch.empty(msda.query_order_workspace_bytes(
                w.B, w.Nq, w.M, w.L, w.P, w.ndim), dtype=torch.uint8, device=dev)
        bufs.append(b)
    stream = torch.cuda.Stream(dev)
    step, launches_per_step = make_step(msda, w, inp, bufs, stream, ordered=args.order,
                                        prune=args.prune, fused=args.fused)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    torch.cuda.synchronize(dev)

    # The K timed steps are captured into one CUDA graph (the library call enqueues plain
    # kernel launches on the given stream, so it is capturable): replaying it issues the
    # launches back to back, so host-side call overhead does not hide kernel time.  The
    # graph is replayed once untimed (upload), then once inside the timed region.
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        graph.capture_begin()
        for i in range(args.steps):
            step(args.warmup + i)
        graph.capture_end()
    with torch.cuda.stream(stream):
        graph.replay()
    torch.cuda.synchronize(dev)

    # Pre-heat: the step graph replayed untimed for about half a second, so that the timed
    # replays start from steady clocks and power state (a few milliseconds of work right
    # after an idle period measured 10-20% slower per step than the steady state).
    t_heat = time.perf_counter()
    while time.perf_counter() - t_heat < args.preheat_s:
        with torch.cuda.stream(stream):
            for _ in range(10):           # back to back: no idle gap between replays
                graph.replay()
        torch.cuda.synchronize(dev)

    # Timed: `replays` separate timings of exactly K steps (one replay of the K-step graph
    # each), every one bracketed by a barrier and a device synchronize; the reported time
    # is the median of the per-rank maxima.  Clocks are sampled over all of them.  Inside
    # each synchronized region one untimed replay runs first, so that the timed steps do
    # not start on a GPU that has just idled through the host's synchronisation (skipped
    # when K is smaller than the number of input sets: the lead-in's inputs would still be
    # in L2 when the timed steps read them again).
    clocks = ClockSampler(local, pci_bus_id(dev))
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    t_replays = []
    lead_in = args.steps >= n_sets
    with clocks:
        for _ in range(args.replays):
            barrier(world)
            torch.cuda.synchronize(dev)
            with torch.cuda.stream(stream):
                if lead_in:
                    graph.replay()
            ev0.record(stream)
            with torch.cuda.stream(stream):
                graph.replay()
            ev1.record(stream)
            clocks.sample_once()
            torch.cuda.synchronize(dev)
            barrier(world)
            t_replays.append(all_max(ev0.elapsed_time(ev1) / 1e3, world))
    t_rank = statistics.median(t_replays)                     # seconds (max over ranks)
    value, t_max = aggregate(t_rank, w.samples, args.steps, world)
    ms_per_step = t_max * 1e3 / args.steps

    # Warm-L2 figure, reported beside the cold one: the same step back to back on one
    # input set, so whatever part of the set fits in L2 stays there between steps.
    n_warm = min(args.steps, 500)
    warm_graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        warm_graph.capture_begin()
        for _ in range(n_warm):
            step(0)
        warm_graph.capture_end()
        warm_graph.replay()
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        warm_graph.replay()               # untimed lead-in, as for the timed replays
    ev0.record(stream)
    with torch.cuda.stream(stream):
        warm_graph.replay()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    t_warm = ev0.elapsed_time(ev1) / 1e3

    # end to end through the public binding, host buffers, copies inside the timed region
    e2e = run_e2e(msda, w, inp, dev, args, world) if not args.no_e2e else None

    if rank != 0:
        barrier(world)
        return None
    byte_inp = fused_byte_inputs(w, inp) if args.fused else inp
    counts = value_row_counts(w, byte_inp)
    ab = algorithmic_bytes(w, byte_inp, counts)
    if args.fused:
        ref_b = inp["reference_points"].nbytes
        ab["total"] += ref_b
        ab["parts"]["reference_points"] = ref_b
        if w.backward:
            ab["total"] += ref_b
            ab["parts"]["grad_reference_points"] = ref_b
    peak, peak_src = measured_peaks()
    per_launch_s = t_rank / args.steps
    achieved = ab["total"] / per_launch_s / 1e9
    mode = ("+order" if args.order == "step" else "+order_once" if args.order == "once" else
            "+fused" if args.fused else
            f"+prune{args.prune:g}" if args.prune > 0 else "")
    traffic = recorded_traffic(w.name, mode)
    clk = clocks.summary()
    secondary = l1_ceiling(w, counts[1], recorded_counter(w.name, mode, "l1_wavefronts_per_launch"),
                           torch.cuda.get_device_properties(dev).multi_processor_count,
                           clk.get("sm_mhz") or clk.get("sm_max_mhz"), per_launch_s,
                           ab["total"], peak)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic",
        "config": run_config(w, args, world),
        "l2_rotation": f"{n_sets} rotating input sets of {set_bytes / 1e6:.1f} MB against "
                       f"{l2 / 2**20:.0f} MiB of L2",
        "hbm_gbs": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_src == "measured" else "fallback 6.4 TB/s",
                     "secondary": secondary,
                     **({"reductions": l2_reduction_ceiling(w, counts[1], per_launch_s)}
                        if w.backward else {}),
                     "nominal": {"peak": NOMINAL_HBM_GBS, "frac": achieved / NOMINAL_HBM_GBS,
                                 "note": "HBM3e nominal, the metric's ~8 TB/s"},
                     "algorithmic_bytes_per_launch": ab["total"],
                     "bytes_breakdown": ab["parts"],
                     "kernel": ("query order + ordered msda fwd" if args.order == "step" else
                                "ordered msda fwd (order computed once per input set)"
                                if args.order == "once" else
                                "pruned msda fwd" if args.prune > 0 else
                                "fused-prologue msda fwd" if args.fused else "msda fwd")
                               if not w.backward else
                               ("zero-fill + fused-prologue msda bwd + epilogues" if args.fused
                                else "query order + zero-fill + ordered msda bwd"
                                if args.order == "step" else
                                "zero-fill + ordered msda bwd (order computed once per input "
                                "set)" if args.order == "once" else "zero-fill + msda bwd")},
        "warm_l2": {"ms_per_step": t_warm * 1e3 / n_warm,
                    "value": w.samples * n_warm / t_warm, "unit": UNIT, "steps": n_warm,
                    "note": "rank 0; one input set back to back, outside the timed region"},
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clk,
        "timing": {"replays": args.replays, "preheat_s": args.preheat_s,
                   "untimed_lead_in_replay": lead_in,
                   "ms_per_step_each": [t * 1e3 / args.steps for t in t_replays],
                   "note": "each timed replay is exactly K steps; ms_per_step is the median"},
        "kernel_source_sha256": kernel_source_hash("backward" if w.backward else "forward"),
    }
    if e2e is not None:
        line["e2e"] = e2e
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, inp, budget_s=args.cpu_budget, fused=args.fused)
    barrier(world)
    return line


def run_e2e(msda, w, inp, dev, args, world):
    """The metric end to end through the public binding: every step uploads its inputs from
    pinned host memory, runs the libmsda call and downloads its result into pinned host
    memory.  Steps are pipelined the way a caller would run a stream of batches: uploads,
    compute and downloads go on three streams, device buffers are double-buffered, so step
    i+1's upload overlaps step i's compute and download (each step still moves all of its
    bytes inside the timed region)."""
    import torch
    pin = {}
    if w.dtype == "bf16":
        pin["value"] = torch.from_numpy(inp["value_bits"].view(np.int16)).view(
            torch.bfloat16).pin_memory()
    else:
        pin["value"] = torch.from_numpy(inp["value"]).pin_memory()
    pin["loc"] = torch.from_numpy(inp["sampling_locations"]).pin_memory()
    pin["attn"] = torch.from_numpy(inp["attention_weights"]).pin_memory()
    if w.backward:
        pin["grad_out"] = (torch.from_numpy(inp["grad_out_bits"].view(np.int16)).view(
            torch.bfloat16) if w.dtype == "bf16" else torch.from_numpy(inp["grad_out"])
        ).pin_memory()
    nbuf = 2
    dins = [{k: torch.empty(v.shape, dtype=v.dtype, device=dev) for k, v in pin.items()}
            for _ in range(nbuf)]
    shapes, starts = inp["spatial_shapes"], inp["level_start_index"]
    if not w.backward:
        fn = msda.msda2d_forward if w.ndim == 2 else msda.msda3d_forward
        out_shapes = [((w.B, w.Nq, w.M * w.D), pin["value"].dtype)]
    else:
        fn = msda.msda2d_backward if w.ndim == 2 else msda.msda3d_backward
        out_shapes = [(tuple(pin["value"].shape), torch.float32),
                      (tuple(pin["loc"].shape), torch.float32),
                      (tuple(pin["attn"].shape), torch.float32)]
    outs_d = [[torch.empty(sh, dtype=dt, device=dev) for sh, dt in out_shapes]
              for _ in range(nbuf)]
    outs_h = [[torch.empty(sh, dtype=dt).pin_memory() for sh, dt in out_shapes]
              for _ in range(nbuf)]
    h2d = sum(v.numel() * v.element_size() for v in pin.values())
    d2h = sum(o.numel() * o.element_size() for o in outs_h[0])
    s_in, s_comp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    in_done = [torch.cuda.Event() for _ in range(nbuf)]
    comp_done = [torch.cuda.Event() for _ in range(nbuf)]
    out_done = [torch.cuda.Event() for _ in range(nbuf)]

    def one(i, compute=True):
        k = i % nbuf
        d, od, oh = dins[k], outs_d[k], outs_h[k]
        if i >= nbuf:
            s_in.wait_event(comp_done[k])       # step i - nbuf no longer reads these inputs
        with torch.cuda.stream(s_in):
            for name in pin:
                d[name].copy_(pin[name], non_blocking=True)
        in_done[k].record(s_in)
        s_comp.wait_event(in_done[k])
        if i >= nbuf:
            s_comp.wait_event(out_done[k])      # step i - nbuf's result has been downloaded
        if not compute:
            pass
        elif not w.backward:
            fn(d["value"], shapes, starts, d["loc"], d["attn"], out=od[0], stream=s_comp)
        else:
            fn(d["value"], shapes, starts, d["loc"], d["attn"], d["grad_out"],
               grad_value=od[0], grad_sampling_locations=od[1], grad_attention_weights=od[2],
               stream=s_comp)
        comp_done[k].record(s_comp)
        s_out.wait_event(comp_done[k])
        with torch.cuda.stream(s_out):
            for o_h, o_d in zip(oh, od):
                o_h.copy_(o_d, non_blocking=True)
        out_done[k].record(s_out)

    steps = max(3, min(args.steps, args.e2e_steps))
    for i in range(3):
        one(i)
    torch.cuda.synchronize(dev)
    barrier(world)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    ev0.record(s_in)
    for i in range(steps):
        one(i)
    ev1.record(s_out)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t0
    t = max(ev0.elapsed_time(ev1) / 1e3, 0.0)
    value, t_max = aggregate(max(t, wall), w.samples, steps, world)
    # The same pipeline with the copies alone (no libmsda call), after the timed region:
    # the floor the host link sets for these bytes (uploads and downloads share it).
    for i in range(3):
        one(i, compute=False)
    torch.cuda.synchronize(dev)
    ev2 = torch.cuda.Event(enable_timing=True)
    ev3 = torch.cuda.Event(enable_timing=True)
    ev2.record(s_in)
    for i in range(steps):
        one(i, compute=False)
    ev3.record(s_out)
    torch.cuda.synchronize(dev)
    copies_ms = ev2.elapsed_time(ev3) / steps
    return {"value": value, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": steps,
            "ms_per_step": t_max * 1e3 / steps,
            "copies_only_ms_per_step": copies_ms,
            "frac_of_copies_only": copies_ms / (t_max * 1e3 / steps),
            "path": "pinned host -> device copies, libmsda call, device -> pinned host "
                    "copies; uploads, compute and downloads on three streams with "
                    "double-buffered device buffers (step i+1 uploads while step i runs)"}


# ----------------------------------------------------------------------------- reference arm


def run_config(w: workloads.Workload, args, world: int) -> dict:
    """The JSON line's `config`: the workload, the mode of the step and how the timing
    treats L2.  Both arms print the same dict for the same command-line flags."""
    return {**workload_config(w),
            "query_order": {"step": "computed each step (msda_query_order) and used by the "
                                    f"ordered {'backward' if w.backward else 'forward'}",
                            "once": "computed once per input set before the timed region "
                                    "(msda_query_order); each step runs the ordered "
                                    f"{'backward' if w.backward else 'forward'}",
                            None: "as given"}[args.order],
            "prologue": ("fused: reference points + pixel offsets + logits in, "
                         "softmax and locations in the kernel") if args.fused
                        else "none: locations and weights given",
            "prune": (f"samples with |A| < {args.prune} skipped: an approximation"
                      if args.prune > 0 else "none (exact)"),
            "l2": "cold: the inputs of consecutive steps rotate over more than twice the "
                  "GPU's L2 capacity",
            "parallelism": f"weak: {world} rank(s), one batch each, no collective"}


def workload_config(w: workloads.Workload) -> dict:
    """The workload keys of the JSON line's `config`, the same on both arms."""
    return {"workload": w.name, "B": w.B, "Nin": w.Nin, "Nq": w.Nq, "M": w.M, "D": w.D,
            "L": w.L, "P": w.P, "levels": [list(s) for s in w.shapes], "ndim": w.ndim,
            "value_dtype": w.dtype, "pass": "backward" if w.backward else "forward",
            "samples_per_step_per_gpu": w.samples}


def run_reference(args):
    """The CPU oracle as it stands, timed on the host cores on this arm's workload and
    metric; each step is a bounded sample (a contiguous block of queries of batch 0)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    import oracle
    oracle.build()
    w = workloads.WORKLOADS[args.workload]
    inp = workloads.make_inputs(w)
    per_q = w.M * w.L * w.P                                  # samples per query
    shapes, starts = inp["spatial_shapes"], inp["level_start_index"]
    value = np.ascontiguousarray(inp["value"][:1], dtype=np.float64)
    loc = np.ascontiguousarray(inp["sampling_locations"][:1], dtype=np.float64)
    attn = np.ascontiguousarray(inp["attention_weights"][:1], dtype=np.float64)
    g = (np.ascontiguousarray(inp["grad_out"][:1], dtype=np.float64) if w.backward else None)

    if args.fused:
        # the fused prologue's inputs: reference points, pixel offsets and logits
        f = workloads.make_fused_inputs(w)
        ref, off, z = (f["reference_points"][:1], f["sampling_offsets"][:1],
                       f["attention_logits"][:1])
        value = np.ascontiguousarray(f["value"][:1], dtype=np.float64)

    # the forward on every host thread (the oracle's block split over OpenMP threads); the
    # backward's grad_value sums are serial, so it runs on one
    threads = 1 if w.backward else 0
    cores = 1 if w.backward else oracle.default_threads()

    def run(q0, q1):
        sl = slice(q0, q1)
        if args.fused and w.backward:
            oracle.backward_fused(w.ndim, value, shapes, starts, ref[:, sl], off[:, sl],
                                  z[:, sl], g[:, sl])
        elif args.fused:
            oracle.forward_fused(w.ndim, value, shapes, starts, ref[:, sl], off[:, sl], z[:, sl],
                                 threads=threads)
        elif w.backward:
            oracle.backward(w.ndim, value, shapes, starts, loc[:, sl], attn[:, sl], g[:, sl])
        elif args.prune > 0:
            oracle.forward_pruned(w.ndim, value, shapes, starts, loc[:, sl], attn[:, sl],
                                  args.prune, threads=threads)
        else:
            oracle.forward(w.ndim, value, shapes, starts, loc[:, sl], attn[:, sl],
                           threads=threads)

    # calibrate: size one step to ~min(0.5 s, 90 s / (K + W))
    nq = min(w.Nq, 256)
    t0 = time.perf_counter()
    run(0, nq)
    rate_q = nq / max(time.perf_counter() - t0, 1e-6)
    budget = min(0.5, 90.0 / max(1, args.steps + args.warmup))
    nq = int(max(1, min(w.Nq, rate_q * budget)))
    for i in range(args.warmup):
        q0 = (i * nq) % max(1, w.Nq - nq + 1)
        run(q0, q0 + nq)
    t0 = time.perf_counter()
    for i in range(args.steps):
        q0 = (i * nq) % max(1, w.Nq - nq + 1)
        run(q0, q0 + nq)
    el = time.perf_counter() - t0
    v = nq * per_q * args.steps / el
    sample = (f"each step: queries [q0, q0+{nq}) of batch 0 of the {w.name} workload "
              f"({nq * per_q} samples), all heads/levels/points; {cores} thread(s), fp64 oracle"
              + ("; fused prologue (reference points, offsets, logits)" if args.fused else ""))
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": run_config(w, args, world),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


# ----------------------------------------------------------------------------- probes

PROBES = (
    # name, kind, rows in the buffer (128 bytes each), lanes per row, what it measures
    ("gather16_l1", 0, 256, 8, "random 128-B rows, 16-B lanes, 32 KB buffer (L1-resident)"),
    ("gather16_l2", 0, 320_000, 8, "random 128-B rows, 16-B lanes, 41 MB buffer (L2-resident)"),
    ("gather16_hbm", 0, 1 << 24, 8, "random 128-B rows, 16-B lanes, 2.1 GB buffer (HBM)"),
    ("gather32_l1", 1, 256, 4, "random 128-B rows, 32-B lanes, 32 KB buffer (L1-resident)"),
    ("gather32_l2", 1, 320_000, 4, "random 128-B rows, 32-B lanes, 41 MB buffer (L2-resident)"),
    ("gather32_hbm", 1, 1 << 24, 4, "random 128-B rows, 32-B lanes, 2.1 GB buffer (HBM)"),
    ("reduce_l2", 2, 320_000, 8, "red.global.add.v4.f32 of random 128-B rows of a 41 MB buffer"),
    ("reduce_hot247", 2, 247, 8, "red.global.add.v4.f32 of random rows of a 247-row hot set"),
    ("smem_atomic_247", 3, 0, 8, "per-channel shared-memory fp32 atomics into a 247-row tile"),
    ("smem_owner_247", 4, 0, 8, "owner-computes shared-memory row updates (no atomics), "
                                "247-row tile"),
    ("tma_gather_l2", 5, 320_000, 1, "cp.async.bulk of random 128-B rows into shared memory, "
                                     "41 MB buffer"),
    # kind 6: 16 rows per warp and batch, so 2 lanes per row in the rows count
    ("tma_gather4_l2", 6, 320_000, 2, "tensor-copy four-row gathers (tile::gather4) of random "
                                      "128-B rows into shared memory, 4 batches of 16 rows in "
                                      "flight per warp, 41 MB buffer"),
    ("tma_gather4_hbm", 6, 1 << 24, 2, "tensor-copy four-row gathers of random 128-B rows, "
                                       "2.1 GB buffer (HBM)"),
)


def run_probes(args):
    """The on-chip rates the kernels are bound by, measured by libmsda_probes.so: random
    128-byte row gathers, reductions and shared-memory updates; rows per second and rows
    per SM clock.  Prints one JSON line per probe."""
    import ctypes
    import torch
    from scale_deformable_attention_msda3d_b300 import build
    lib = ctypes.CDLL(build.build_probes())
    lib.msda_probe_launch.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_uint, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_uint, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_void_p]
    lib.msda_probe_launch.restype = ctypes.c_int
    lib.msda_probe_block.argtypes = [ctypes.c_int]
    dev = torch.device("cuda", 0)
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    stream = torch.cuda.Stream(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    for name, kind, n_rows, lanes, what in PROBES:
        if args.probe not in ("all", name):
            continue
        threads = lib.msda_probe_block(kind)
        blocks = sms * (2048 // threads)
        buf = torch.zeros(max(n_rows, 1) * 32, dtype=torch.float32, device=dev)
        if kind in (0, 1, 5, 6):
            buf.uniform_()
        sink = torch.empty(blocks * threads, dtype=torch.float32, device=dev)
        iters = 256 if kind != 5 else 64
        rows_per_launch = blocks * threads // lanes * iters

        def launch(seed):
            rc = lib.msda_probe_launch(kind, ctypes.c_void_p(buf.data_ptr()), n_rows, blocks, iters,
                                       seed, ctypes.c_void_p(sink.data_ptr()),
                                       ctypes.c_void_p(err.data_ptr()),
                                       ctypes.c_void_p(stream.cuda_stream))
            if rc != 0:
                raise RuntimeError(f"probe {name}: launch status {rc}")

        for i in range(3):
            launch(i)
        torch.cuda.synchronize(dev)
        times = []
        for r in range(5):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            launch(100 + r)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            times.append(e0.elapsed_time(e1) / 1e3)
        if int(err.item()) != 0:
            raise RuntimeError(f"probe {name}: a bounded wait ran out")
        t = statistics.median(times)
        rate = rows_per_launch / t
        line = {"probe": name, "what": what, "rows_per_s": rate, "row_bytes": 128,
                "bytes_per_s": rate * 128, "rows_per_launch": rows_per_launch,
                "launch_us": t * 1e6, "blocks": blocks, "threads": threads, "sms": sms,
                "rows_per_sm_clock_at_2032mhz": rate / (sms * 2.032e9)}
        print(json.dumps(line), flush=True)
        del buf, sink
    return None


def build_parser() -> argparse.ArgumentParser:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=workloads.names(), default="encoder2d")
    ap.add_argument("--order", nargs="?", const="step", default=None,
                    choices=["step", "once"],
                    help="run the ordered forward (backward workloads: the ordered backward) "
                         "with the locality-aware query order computed inside each step "
                         "('step', the default), or computed once per input set before the "
                         "timed region ('once': an encoder's layers share their reference "
                         "points and can share one order, and a backward can reuse its "
                         "forward's order)")
    ap.add_argument("--fused", action="store_true",
                    help="reference points, pixel offsets and logits in; the kernel forms "
                         "locations and the softmax (backward workloads: the fused backward, "
                         "with offset, logit and reference-point gradients; no e2e leg)")
    ap.add_argument("--prune", type=float, default=0.0,
                    help="forward workloads: skip samples with |A| below this threshold "
                         "(approximate; 0 = exact)")
    ap.add_argument("--replays", type=int, default=5,
                    help="timed replays of the K-step graph (each exactly K steps); the "
                         "median is reported")
    ap.add_argument("--preheat-s", type=float, default=0.5,
                    help="seconds of untimed replays before the timed ones")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle time for the cpu_baseline leg")
    ap.add_argument("--probe", default=None,
                    help="run the on-chip rate microbenchmarks instead of the step ('all' or "
                         "one probe name) and print one JSON line per probe")
    return ap


def main(argv=None):
    ap = build_parser()
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.prune > 0 and workloads.WORKLOADS[args.workload].backward:
        ap.error("--prune applies to the forward workloads")
    if sum([bool(args.order), args.prune > 0, bool(args.fused)]) > 1:
        ap.error("--order, --prune and --fused are separate modes")
    if args.fused:
        args.no_e2e = True
    if args.probe:
        run_probes(args)
        return 0
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)
    if int(os.environ.get("WORLD_SIZE", "1")) > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
