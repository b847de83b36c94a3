#!/usr/bin/env python3
"""Benchmark of the ZVC hot path on the GoogLeNet-shaped activation batch.

One step is the whole device path on the 57 GoogLeNet-shaped activation tensors at batch
256 (3,020,193,792 fp32 words, 12.1 GB, 5-60% non-zero): one zvc_compress_batched launch
over all 57 tensors (zero test, masks, popcounts, offsets, packing: Rhu et al.,
"Compressing DMA Engine", section V.A; offsets from prefix sums, section V.B), then one
zvc_decompress_batched launch that restores them. `value` is the slower kernel's
uncompressed GB/s (4n bytes per launch over its device time), with the activations in HBM.

The same line reports, measured in the same run:
  compress / decompress   each kernel's uncompressed GB/s, its algorithmic HBM bytes
                (4n read + S written, S read + 4n written) per second and their fraction
                of the measured HBM copy bandwidth
  roofline      the slower (dominant) kernel's algorithmic bytes per launch over its
                launch time (CUDA events bracketing that one launch on its stream)
  e2e           the same metric through the offload/prefetch calls with the activations
                in pinned host memory (section V.D: offload and prefetch with
                cudaMemcpyAsync): H2D of the inputs + zvc_offload (compress, D2H of the
                compressed segments), then zvc_prefetch (H2D, decompress) + D2H of the
                restored tensors; the slower direction's uncompressed GB/s, median of the
                repetitions, beside plain copies of the same bytes taken after each one
  alexnet_stack the offload/prefetch step on the 5-layer AlexNet stack (333 MB) with its
                host-link figures, and each kernel on those layers
  cpu_baseline  the single-threaded CPU oracle on a bounded sample of the same workload
`--impl reference` times that oracle alone (the pages describe hardware; the oracle is
the only other implementation of this path).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "ZVC compress/decompress GB/s (uncompressed) and % of HBM roofline; ratio"
WORKLOAD = ("googlenet_batch: 57 GoogLeNet-shaped fp32 activation tensors at batch 256 "
            "(spatial 112/56/28/14/7, 64-1024 channels, 3,020,193,792 words = 12.1 GB), each "
            "ReLU(x - Phi^-1(1 - d_i)), x ~ N(0,1), d_i ~ U[5%, 60%]; one batched launch each way")
ALEXNET_WORKLOAD = ("alexnet_stack: batch-128 AlexNet conv activations 96x55x55, 256x27x27, "
                    "384x13x13, 384x13x13, 256x13x13 fp32 = ReLU(x + b_c), non-zero "
                    "60/45/35/30/20%")
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0  # the vendor's HBM3e figure for GB300: context only, labelled as such
SAMPLE_BATCH = 2  # CPU oracle sample: the GoogLeNet batch at batch 2 (1/128 of batch 256)


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--chunk-elems", type=int, default=4096)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--profile", choices=["compress", "decompress", "compress_batch",
                                          "decompress_batch"],
                   help="run a few launches of one kernel and exit: compress/decompress on "
                        "AlexNet layer 0 (149 MB), *_batch on the GoogLeNet batch at "
                        "--profile-batch (the small case for ncu captures)")
    p.add_argument("--profile-batch", type=int, default=16, metavar="B",
                   help="with --profile *_batch: the GoogLeNet batch at batch B (16: 755 MB)")
    p.add_argument("--no-context", action="store_true",
                   help="skip the AlexNet-stack context measurements (for launch lists)")
    p.add_argument("--profile-density", type=float, default=None, metavar="D",
                   help="with --profile: a flat map of the same size with a fraction D of "
                        "i.i.d. non-zero words, instead of AlexNet layer 0")
    p.add_argument("--profile-layer", type=int, default=0, metavar="L",
                   help="with --profile compress|decompress: AlexNet layer L (0-4) of the "
                        "batch-128 stack instead of layer 0")
    p.add_argument("--train", action="store_true",
                   help="training step of a VGG-style CNN with its saved activations kept, "
                        "offloaded compressed to host memory, or kept compressed in HBM; "
                        "prints one JSON line and exits")
    p.add_argument("--layouts", action="store_true",
                   help="ZVC and RLE compression ratios of the AlexNet stack and the VGG "
                        "conv1_2 map in NCHW, NHWC and CHWN, and RLE kernel times; prints "
                        "one JSON line and exits")
    p.add_argument("--configs", action="store_true",
                   help="both kernels on every input configuration (single map, AlexNet "
                        "layers, VGG conv1_2, the 2^28-word density sweep, the 57-tensor "
                        "GoogLeNet batch in one batched launch each way); prints one JSON "
                        "line and exits")
    p.add_argument("--configs16", action="store_true",
                   help="the 16-bit calls (zvc_compress16 / zvc_decompress16) on bf16 copies of "
                        "the single-tensor configurations (AlexNet layers, VGG conv1_2, the "
                        "2^28-word density sweep); prints one JSON line and exits")
    p.add_argument("--write-traffic", nargs=2, metavar=("COMPRESS_CSV", "DECOMPRESS_CSV"),
                   help="turn ncu DRAM counters of one step's launches (see TRAFFIC_FILE) "
                        "into that file, keyed by the kernels' source hashes, and exit")
    return p.parse_args(argv)


# ------------------------------------------------------------------ DRAM traffic record
# `traffic` in the bench line comes from ncu counters taken on the step's kernels: the
# dram__bytes_read.sum + dram__bytes_write.sum of one zvc_compress_batched and one
# zvc_decompress_batched launch on the GoogLeNet batch at batch B (755 MB of input at the
# default B = 16, larger than the 129 MB L2, a few GB on the device), captured with
#   ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum
#       --clock-control none -k regex:^<kernel> -s 1 -c 1 --csv --log-file <csv>
#       python bench.py --profile <compress|decompress>_batch --profile-batch B
# (the second launch of the kernel in that run; the first is a warm-up). Every word is
# read (written) once and every stream byte written (read) once, so a launch moves the
# same bytes per word at any batch: the record holds bytes per word and the hash of the
# kernel's sources, and the line scales it by the words of one full-size launch. Once a
# source changes the record no longer applies and `traffic` is null until it is captured
# again.
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "step_traffic.json")
KERNEL_SOURCES = {
    "compress_kernel": ["zvc_compress.cu", "zvc_internal.cuh"],
    "decompress_kernel": ["zvc_decompress.cu", "zvc_plan.h", "zvc_internal.cuh"],
}


def kernel_source_hash(kernel: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "activation_sparsity_compression_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def ncu_csv_metrics(csv_path: str):
    """Per launch (in capture order) a dict of metric name -> value in base units (bytes,
    nanoseconds) from an ncu --csv log."""
    import csv
    rows = list(csv.reader(open(csv_path)))
    h = next(i for i, r in enumerate(rows) if r and r[0] == "ID")
    hdr = rows[h]
    ii, mi, vi, ui = (hdr.index(x) for x in ("ID", "Metric Name", "Metric Value", "Metric Unit"))
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9,
             "ns": 1, "nsecond": 1, "usecond": 1e3, "us": 1e3, "msecond": 1e6, "ms": 1e6}
    per = {}
    for r in rows[h + 1:]:
        if len(r) > vi and r[mi]:
            v = float(r[vi].replace(",", "")) * scale.get(r[ui], 1)
            per.setdefault(r[ii], {})[r[mi]] = v
    return [per[k] for k in sorted(per, key=int)]


def ncu_dram_bytes(csv_path: str):
    """Per-launch dram__bytes_read.sum + dram__bytes_write.sum from an ncu --csv log."""
    return [m.get("dram__bytes_read.sum", 0.0) + m.get("dram__bytes_write.sum", 0.0)
            for m in ncu_csv_metrics(csv_path)]


def write_traffic(csvs, chunk_elems, batch):
    import workloads
    import math
    n_words = sum(math.prod(s.shape) for s in workloads.googlenet_specs(batch))
    rec = {"command": "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,"
                      "gpu__time_duration.sum --clock-control none -k regex:^<kernel> -s 1 "
                      "-c 1 --csv --log-file <csv> python bench.py --profile <kernel>_batch "
                      f"--profile-batch {batch}",
           "workload": f"googlenet batch at batch {batch}", "words_per_launch": n_words,
           "chunk_elems": chunk_elems, "kernels": {}}
    for kernel, path in zip(("compress_kernel", "decompress_kernel"), csvs):
        ms = ncu_csv_metrics(path)
        if len(ms) != 1:
            raise SystemExit(f"{path}: {len(ms)} launches captured, expected 1")
        b = ms[0].get("dram__bytes_read.sum", 0.0) + ms[0].get("dram__bytes_write.sum", 0.0)
        rec["kernels"][kernel] = {"source_sha256": kernel_source_hash(kernel),
                                  "dram_bytes": b, "dram_bytes_per_word": b / n_words,
                                  "gpu_time_us": ms[0].get("gpu__time_duration.sum", 0.0) / 1e3}
    with open(TRAFFIC_FILE, "w") as f:
        json.dump(rec, f, indent=1)
    print(json.dumps(rec))
    return 0


def traffic_per_launch(kernel: str, words_per_launch: float):
    """DRAM bytes one launch of `kernel` moves at this size, from the record, or None."""
    try:
        rec = json.load(open(TRAFFIC_FILE))["kernels"][kernel]
    except (OSError, KeyError, ValueError):
        return None
    if rec.get("source_sha256") != kernel_source_hash(kernel):
        return None
    return rec["dram_bytes_per_word"] * words_per_launch


# ------------------------------------------------------------------ multi-rank plumbing
def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def dist_init(backend):
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)
    return rank, world, local


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def reduce_max(v: float, device=None) -> float:
    """Maximum of v over ranks (v itself with one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(v)
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_rank_per_step: float, world: int, steps: int, max_ms: float) -> float:
    """Units all ranks processed divided by the slowest rank's time, in GB/s."""
    return bytes_per_rank_per_step * world * steps / (max_ms / 1e3) / 1e9


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_uuid):
        self.uuid = gpu_uuid
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "50"]
        if self.uuid:
            cmd.insert(1, f"--id={self.uuid}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"),
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts, float(parts[1]), float(parts[2]), parts[4:]))
            except (ValueError, IndexError):
                continue
        os.unlink(self.path)
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        if not inside and rows:  # a timed region shorter than the sampling period
            inside = [min(rows, key=lambda r: abs(r[0] - (t0 + t1) / 2))]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = set()
        for r in inside:
            for name, val in zip(names[1:], r[3][1:]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "samples": len(inside),
                "reasons": sorted(reasons)}


class NvmlSampler:
    """Samples the SM clock, its maximum and the clock event (throttle) reasons through
    NVML every few milliseconds on a thread, so that a timed region of a hundred
    milliseconds still gets tens of samples. Reads only; changes no setting. Falls back to
    ClockSampler (nvidia-smi) where NVML cannot be loaded."""
    NVML_CLOCK_SM = 1
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu_uuid, period_s=0.005):
        self.uuid = gpu_uuid
        self.period = period_s
        self.rows = []
        self.thread = None
        self.stop_flag = threading.Event()
        self.lib = self.dev = self.reason_fn = None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            dev = ctypes.c_void_p()
            if not gpu_uuid or lib.nvmlDeviceGetHandleByUUID(gpu_uuid.encode(),
                                                             ctypes.byref(dev)) != 0:
                return
            for name in ("nvmlDeviceGetCurrentClocksEventReasons",
                         "nvmlDeviceGetCurrentClocksThrottleReasons"):
                if hasattr(lib, name):
                    self.reason_fn = getattr(lib, name)
                    break
            self.lib, self.dev = lib, dev
        except OSError:
            pass

    def available(self):
        return self.lib is not None and self.reason_fn is not None

    def _sample(self):
        sm, mx = ctypes.c_uint(), ctypes.c_uint()
        r = ctypes.c_ulonglong()
        if (self.lib.nvmlDeviceGetClockInfo(self.dev, self.NVML_CLOCK_SM, ctypes.byref(sm)) or
                self.lib.nvmlDeviceGetMaxClockInfo(self.dev, self.NVML_CLOCK_SM, ctypes.byref(mx)) or
                self.reason_fn(self.dev, ctypes.byref(r))):
            return None
        return time.time(), float(sm.value), float(mx.value), int(r.value)

    def _run(self):
        while not self.stop_flag.is_set():
            row = self._sample()
            if row:
                self.rows.append(row)
            time.sleep(self.period)

    def start(self):
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()
        time.sleep(0.05)

    def stop(self, t0, t1):
        self.stop_flag.set()
        self.thread.join()
        inside = [r for r in self.rows if t0 <= r[0] <= t1]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "source": "nvml"}
        reasons = sorted({name for r in inside for bit, name in self.REASONS.items() if r[3] & bit})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "samples": len(inside),
                "reasons": reasons, "source": "nvml, 5 ms period"}


def clock_sampler(gpu_uuid):
    s = NvmlSampler(gpu_uuid)
    return s if s.available() else ClockSampler(gpu_uuid)


def host_cpu():
    """(logical cores this process may use, CPU model) of the host."""
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count() or 1
    model = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() == "Model name":
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    return cores, f"{model or platform.processor() or 'unknown'} ({platform.machine()})"


# ------------------------------------------------------------------ CPU oracle leg
def oracle_sample(chunk_elems: int, budget_s: float, batch: int = SAMPLE_BATCH):
    """Times the CPU oracle on the GoogLeNet batch generated at a reduced batch: encode
    (compress) and decode (decompress) of every tensor, timed apart, passing over the
    sample until budget_s of CPU work is done (at least one whole pass; the first pass is
    checked bit-exact). Returns (encode GB/s, decode GB/s, words, seconds, passes), in
    uncompressed bytes."""
    import numpy as np

    import oracle
    import workloads

    lib = oracle.load()
    tensors = [x.numpy().view(np.uint32).reshape(-1) for x in
               workloads.googlenet_batch(device="cpu", batch=batch)]
    te = td = 0.0
    done = passes = 0
    while True:
        for w in tensors:
            t0 = time.perf_counter()
            s = oracle.encode(w, chunk_elems, lib=lib)
            t1 = time.perf_counter()
            st, back = oracle.decode(s, w.size, chunk_elems, lib=lib)
            t2 = time.perf_counter()
            te += t1 - t0
            td += t2 - t1
            if st != oracle.OK or (passes == 0 and not np.array_equal(back, w)):
                raise RuntimeError("oracle round trip failed")
            done += w.size
        passes += 1
        if te + td > budget_s:
            break
    return 4 * done / te / 1e9, 4 * done / td / 1e9, done, te + td, passes


def cpu_baseline_record(chunk_elems: int, budget_s: float):
    enc, dec, words, secs, passes = oracle_sample(chunk_elems, budget_s)
    cores, model = host_cpu()
    return {"value": min(enc, dec), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "encode_gbs": enc, "decode_gbs": dec, "host_cores": cores, "cpu_model": model,
            "sample": f"googlenet_batch at batch {SAMPLE_BATCH} (1/{256 // SAMPLE_BATCH} of "
                      f"batch 256, the same 57 shapes and densities), {passes} passes: {words} "
                      f"words encoded and decoded in {secs:.1f} s on one thread; value = the "
                      "slower of encode and decode, as on the GPU line"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import numpy as np

    import oracle
    import workloads

    lib = oracle.load()
    tensors = [x.numpy().view(np.uint32).reshape(-1) for x in
               workloads.googlenet_batch(device="cpu", batch=SAMPLE_BATCH)]
    n = sum(w.size for w in tensors)
    tally = [0.0, 0.0]

    def step():
        for w in tensors:
            t0 = time.perf_counter()
            s = oracle.encode(w, args.chunk_elems, lib=lib)
            t1 = time.perf_counter()
            st, _ = oracle.decode(s, w.size, args.chunk_elems, lib=lib)
            t2 = time.perf_counter()
            tally[0] += t1 - t0
            tally[1] += t2 - t1
            if st != oracle.OK:
                raise RuntimeError("oracle decode failed")

    for _ in range(args.warmup):
        step()
    tally[0] = tally[1] = 0.0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    enc = 4 * n * args.steps / tally[0] / 1e9
    dec = 4 * n * args.steps / tally[1] / 1e9
    value = min(enc, dec)
    cores, model = host_cpu()
    sample = (f"googlenet_batch at batch {SAMPLE_BATCH} (1/{256 // SAMPLE_BATCH} of batch 256, "
              f"{n} words, the same 57 shapes and densities) per step; oracle encode and "
              "decode of every tensor, single thread")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "chunk_elems": args.chunk_elems,
                       "sample_batch": SAMPLE_BATCH,
                       "value": "the slower of encode and decode, uncompressed GB/s"},
            "compress": {"gbs": enc}, "decompress": {"gbs": dec},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "host_cores": cores, "cpu_model": model, "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU leg
def _uuid(torch, dev):
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        return None


def run_ours(args):
    import torch

    rank, world, local = dist_init("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from activation_sparsity_compression_gb300 import build as zbuild
    zbuild.build()
    import activation_sparsity_compression_gb300 as zvc
    import workloads

    C = args.chunk_elems
    K = args.steps
    xs = workloads.googlenet_batch(device=dev)
    ns = [x.numel() for x in xs]
    N = sum(ns)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    def ok(st, where):
        if st != zvc.ZVC_OK:
            raise zvc.ZvcError(st, where)

    cap = zvc.zvc_batch_size_bound(ns, C)
    out = torch.empty(cap, dtype=torch.uint8, device=dev)
    size = torch.zeros(1, dtype=torch.int64, device=dev)
    ws = zvc.new_workspace(max(zvc.zvc_batch_workspace_size(ns, C), 256), dev)
    ys = [torch.empty_like(x) for x in xs]
    xp, yp = [x.data_ptr() for x in xs], [y.data_ptr() for y in ys]
    S_box = [0]

    def comp():
        ok(zvc.zvc_compress_batched(xp, ns, C, out.data_ptr(), cap, size.data_ptr(),
                                    ws.data_ptr(), ws.numel(), sh), "zvc_compress_batched")

    def decomp():
        ok(zvc.zvc_decompress_batched(out.data_ptr(), S_box[0], yp, ns, C, ws.data_ptr(),
                                      ws.numel(), sh), "zvc_decompress_batched")

    def check(where):
        ok(zvc.zvc_get_error(ws.data_ptr(), sh), where)
        if int(size.item()) != S_box[0]:
            raise RuntimeError(f"{where}: stream size changed")
        for i, (x, y) in enumerate(zip(xs, ys)):
            if not torch.equal(x.view(torch.int32), y.view(torch.int32)):
                raise RuntimeError(f"{where}: tensor {i} is not restored bit-exactly")

    comp()
    torch.cuda.synchronize(dev)
    S_box[0] = S = int(size.item())
    for _ in range(max(args.warmup, 1)):
        comp()
        decomp()
    torch.cuda.synchronize(dev)
    check("warm-up")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = clock_sampler(_uuid(torch, dev))
    sampler.start()
    barrier()
    torch.cuda.synchronize(dev)
    w0 = time.time()
    e_start.record(stream)
    for k in range(K):
        ev[k][0].record(stream)
        comp()
        ev[k][1].record(stream)
        decomp()
        ev[k][2].record(stream)
    e_end.record(stream)
    torch.cuda.synchronize(dev)
    w1 = time.time()
    barrier()
    clocks = sampler.stop(w0, w1)
    check("timed steps")
    ms = reduce_max(e_start.elapsed_time(e_end), dev)
    lc = [e[0].elapsed_time(e[1]) for e in ev]  # this rank's launch times, ms
    ld = [e[1].elapsed_time(e[2]) for e in ev]
    tc = reduce_max(sum(lc), dev)
    td = reduce_max(sum(ld), dev)
    peak, peak_kind = hbm_peak()
    moved = 4 * N + S

    def kernel_rec(t, launches):
        return {"gbs": whole_job_gbs(4 * N, world, K, t),
                "hbm_gbs": whole_job_gbs(moved, world, K, t),
                "hbm_frac": whole_job_gbs(moved, world, K, t) / peak / world,
                "hbm_frac_of_nominal": whole_job_gbs(moved, world, K, t) / NOMINAL_HBM_GBS / world,
                "launches": K, "avg_launch_us": t / K * 1e3,
                "median_launch_us": statistics.median(launches) * 1e3,
                "best_launch_us": min(launches) * 1e3}

    comp_rec, decomp_rec = kernel_rec(tc, lc), kernel_rec(td, ld)
    value = min(comp_rec["gbs"], decomp_rec["gbs"])
    kern, t = ("compress", tc) if tc >= td else ("decompress", td)
    achieved = moved / (t / K / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": f"{kern}_kernel", "achieved": achieved, "peak": peak,
                "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                "traffic": traffic_per_launch(f"{kern}_kernel", N),
                "traffic_unit": "bytes per launch",
                "algorithmic_bytes_per_launch": moved, "avg_launch_us": t / K * 1e3,
                "timing": "CUDA events on the launching stream bracketing each launch",
                "share_of_step": t / ms,
                "kernels": {"compress_kernel": {"launches": K, "ms": tc, "share_of_step": tc / ms},
                            "decompress_kernel": {"launches": K, "ms": td,
                                                  "share_of_step": td / ms}}}

    del ev
    e2e = measure_e2e_batch(args, zvc, torch, xs, ys, ns, C, dev, stream)

    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": ms / K,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "tensors": len(ns), "n_words": N,
                       "chunk_elems": C,
                       "step": "zvc_compress_batched over the 57 tensors, then "
                               "zvc_decompress_batched back (one launch each)",
                       "value": "the slower kernel's uncompressed GB/s (4n bytes per launch "
                                "over its device time)",
                       "l2": "inputs larger than L2 (12.1 GB per launch), no flush"},
            "ratio": 4 * N / S, "stream_bytes": S,
            "compress": comp_rec, "decompress": decomp_rec,
            "roofline": roofline, "gpu_launches": 2 * K, "clocks": clocks, "e2e": e2e}
    if not args.no_context:
        line["alexnet_stack"] = alexnet_context(args, zvc, torch, dev, stream, peak)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_record(C, 12.0)
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


class PinnedSlab:
    """Page-locked host buffers of the given byte sizes, carved at 256-byte boundaries out
    of one torch pinned allocation (cudaHostAlloc). One slab rather than one allocation per
    tensor: torch's pinned allocator rounds every block up to a power of two. (An earlier
    version registered 114 separate buffers, 24 GB in all, with cudaHostRegister; its
    step ran at 12-13 GB/s, although 1 GB registered alone copies at 190 GB/s. The cause
    was not isolated.)"""
    def __init__(self, torch, sizes):
        offs, pos = [], 0
        for n in sizes:
            offs.append(pos)
            pos += -(-int(n) // 256) * 256
        self.buf = torch.empty(max(pos, 256), dtype=torch.uint8, pin_memory=True)
        self.views = [self.buf[o:o + int(n)] for o, n in zip(offs, sizes)]


def measure_e2e_batch(args, zvc, torch, xs, ys, ns, C, dev, stream):
    """The same metric through the public offload/prefetch calls with the activations in
    pinned host memory. Per step: the H2D copy of every tensor (a copy stream) and its
    zvc_offload (compress, D2H of the compressed segments), then zvc_prefetch (H2D of the
    segments, decompress) and the D2H copy of every restored tensor back into the same
    pinned buffers (a second copy stream). The two directions are timed apart with events
    on the caller's stream, each repetition on its own; the value is the slower direction's
    uncompressed GB/s over the median repetition."""
    sh = stream.cuda_stream
    T = len(xs)
    N = sum(ns)
    slab_x = PinnedSlab(torch, [4 * n for n in ns])
    hx = [v.view(torch.float32) for v in slab_x.views]
    for h, x in zip(hx, xs):
        h.copy_(x.view(-1))
    dx = [torch.empty(n, dtype=torch.float32, device=dev) for n in ns]
    hcap = [zvc.zvc_offload_host_bound(n, C) for n in ns]
    hb = PinnedSlab(torch, hcap).views
    ows = zvc.new_workspace(max(zvc.zvc_offload_workspace_size(n, C) for n in ns), dev)
    hs = [0] * T
    cin, cout = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(T)]
    ev_out = [torch.cuda.Event() for _ in range(T)]

    def ok(st, where):
        if st != zvc.ZVC_OK:
            raise zvc.ZvcError(st, where)

    def offload_dir():
        cin.wait_stream(stream)
        with torch.cuda.stream(cin):
            for i in range(T):
                dx[i].copy_(hx[i], non_blocking=True)
                ev_in[i].record(cin)
        for i in range(T):
            stream.wait_event(ev_in[i])
            st, hs[i] = zvc.zvc_offload(dx[i].data_ptr(), ns[i], C, hb[i].data_ptr(), hcap[i],
                                        ows.data_ptr(), ows.numel(), sh)
            ok(st, "zvc_offload")
        ok(zvc.zvc_offload_join(sh), "zvc_offload_join")

    def prefetch_dir():
        for i in range(T):
            ok(zvc.zvc_prefetch(hb[i].data_ptr(), hs[i], ys[i].data_ptr(), ns[i], C,
                                ows.data_ptr(), ows.numel(), sh), "zvc_prefetch")
            ev_out[i].record(stream)
            cout.wait_event(ev_out[i])
            with torch.cuda.stream(cout):
                hx[i].copy_(ys[i].view(-1), non_blocking=True)
        stream.wait_stream(cout)

    for _ in range(2):
        offload_dir()
        prefetch_dir()
    torch.cuda.synchronize(dev)
    ok(zvc.zvc_get_error(ows.data_ptr(), sh), "e2e warm-up")
    for i, (x, y) in enumerate(zip(xs, ys)):
        if not torch.equal(x.view(torch.int32), y.view(torch.int32)):
            raise RuntimeError(f"e2e: tensor {i} is not restored bit-exactly")
    _, world, _ = dist_env()
    segs = [-(-n // zvc.zvc_offload_segment_elems(n, C)) for n in ns]
    link = sum(h - (16 + 8 * (k + 1)) for h, k in zip(hs, segs))  # segment streams moved

    # The floor each direction has on this host link: plain copies of the same bytes, the
    # two ways at once as in the step (offload: the inputs in, the compressed bytes out;
    # prefetch: the compressed bytes in, the restored tensors out), with no kernel between.
    # It is taken right after each repetition of the step, so that both see the same load
    # on the host link (the link is shared with the machine's other GPUs and their jobs,
    # whose traffic comes and goes). The floor's copies overwrite the host streams and the
    # device inputs, which the next repetition writes again before it reads them, and copy
    # the restored tensors back over the host inputs, which they equal.
    yb = [y.view(-1).view(torch.uint8) for y in ys]
    xb = [x.view(torch.uint8) for x in dx]
    kb = [min(h, 4 * n) for h, n in zip(hs, ns)]  # the compressed bytes (of a device buffer)
    off_pairs = ([(dx[i], hx[i]) for i in range(T)],
                 [(hb[i][:kb[i]], yb[i][:kb[i]]) for i in range(T)])
    pre_pairs = ([(xb[i][:kb[i]], hb[i][:kb[i]]) for i in range(T)],
                 [(hx[i], ys[i].view(-1)) for i in range(T)])

    def floor_ms(h2d, d2h):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for st, pairs in ((cin, h2d), (cout, d2h)):
            st.wait_stream(stream)
            with torch.cuda.stream(st):
                for dst, src in pairs:
                    dst.copy_(src, non_blocking=True)
        stream.wait_stream(cin)
        stream.wait_stream(cout)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1)

    reps = max(5, min(args.steps, 9))
    t_in, t_out, f_in, f_out = [], [], [], []
    barrier()
    torch.cuda.synchronize(dev)
    for _ in range(reps):
        m = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        m[0].record(stream)
        offload_dir()
        m[1].record(stream)
        prefetch_dir()
        m[2].record(stream)
        torch.cuda.synchronize(dev)
        t_in.append(m[0].elapsed_time(m[1]))
        t_out.append(m[1].elapsed_time(m[2]))
        ok(zvc.zvc_get_error(ows.data_ptr(), sh), "e2e")
        for i, (x, y) in enumerate(zip(xs, ys)):
            if not torch.equal(x.view(torch.int32), y.view(torch.int32)):
                raise RuntimeError(f"e2e: tensor {i} is not restored bit-exactly")
        f_in.append(floor_ms(*off_pairs))
        f_out.append(floor_ms(*pre_pairs))
    for i, (h, x) in enumerate(zip(hx, xs)):  # the host copies, once
        if not torch.equal(h.view(torch.int32), x.view(-1).view(torch.int32).cpu()):
            raise RuntimeError(f"e2e: host tensor {i} is not restored bit-exactly")

    def gbs(ms):  # uncompressed GB/s of one step that took ms
        return whole_job_gbs(4 * N, world, 1, reduce_max(ms, dev))

    med = statistics.median
    off_gbs, pre_gbs = gbs(med(t_in)), gbs(med(t_out))
    off_floor, pre_floor = gbs(med(f_in)), gbs(med(f_out))
    return {"value": min(off_gbs, pre_gbs), "unit": "GB/s",
            "statistic": "median of the repetitions (each direction)",
            "h2d_bytes_per_step": 4 * N + link,
            "d2h_bytes_per_step": link + 8 * sum(segs) + 4 * N,
            "steps": reps, "offload_direction_gbs": off_gbs, "prefetch_direction_gbs": pre_gbs,
            "best_gbs": min(gbs(min(t_in)), gbs(min(t_out))),
            "mean_gbs": min(gbs(sum(t_in) / reps), gbs(sum(t_out) / reps)),
            "offload_direction_ms": t_in, "prefetch_direction_ms": t_out,
            "compressed_link_bytes_per_direction": link,
            "link_floor": {"offload_direction_gbs": off_floor,
                           "prefetch_direction_gbs": pre_floor,
                           "offload_direction_ms": f_in, "prefetch_direction_ms": f_out,
                           "frac_of_floor": min(off_gbs, pre_gbs) / min(off_floor, pre_floor),
                           "what": "plain pinned cudaMemcpyAsync of the same bytes, both ways "
                                   "at once as in each direction of the step, no kernels, "
                                   "right after each repetition; uncompressed GB/s, median"},
            "call": "H2D copy + zvc_offload per tensor, zvc_offload_join; zvc_prefetch + "
                    "D2H copy per tensor"}


def alexnet_context(args, zvc, torch, dev, stream, peak):
    """The offload/prefetch step on the AlexNet stack (every layer offloaded, then
    prefetched in reverse order, as vDNN does), its host-link figures, and each kernel on
    those layers alone (one launch per layer, and one batched launch over the stack)."""
    import workloads

    C = args.chunk_elems
    xs = workloads.alexnet_stack(device=dev)
    ns = [x.numel() for x in xs]
    N = sum(ns)
    L = len(xs)
    sh = stream.cuda_stream
    hcap = [zvc.zvc_offload_host_bound(n, C) for n in ns]
    hbuf = [torch.empty(c, dtype=torch.uint8, pin_memory=True) for c in hcap]
    ws = [zvc.new_workspace(zvc.zvc_offload_workspace_size(n, C), dev) for n in ns]
    ys = [torch.empty_like(x) for x in xs]
    hsize = [0] * L

    def step():
        for l in range(L):
            st, hsize[l] = zvc.zvc_offload(xs[l].data_ptr(), ns[l], C, hbuf[l].data_ptr(),
                                           hcap[l], ws[l].data_ptr(), ws[l].numel(), sh)
            if st != zvc.ZVC_OK:
                raise zvc.ZvcError(st, "zvc_offload")
        for l in reversed(range(L)):
            st = zvc.zvc_prefetch(hbuf[l].data_ptr(), hsize[l], ys[l].data_ptr(), ns[l], C,
                                  ws[l].data_ptr(), ws[l].numel(), sh)
            if st != zvc.ZVC_OK:
                raise zvc.ZvcError(st, "zvc_prefetch")

    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    for l in range(L):
        if zvc.zvc_get_error(ws[l].data_ptr(), sh) != zvc.ZVC_OK or not torch.equal(
                xs[l].view(torch.int32), ys[l].view(torch.int32)):
            raise RuntimeError(f"alexnet step: layer {l} is not restored bit-exactly")
    reps = 20
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(reps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1)
    res = {"workload": ALEXNET_WORKLOAD, "n_words": N,
           "offload_prefetch_step": {"gbs": 4 * N * reps / (ms / 1e3) / 1e9,
                                     "ms_per_step": ms / reps,
                                     "link_bytes_per_direction": sum(hsize),
                                     "step": "zvc_offload of 5 layers, then zvc_prefetch in "
                                             "reverse order"}}
    res.update(measure_components(args, zvc, torch, xs, ns, C, dev, stream, peak))
    return res


def _trace(zvc, fn):
    zvc.zvc_trace_start()
    fn()
    st, t = zvc.zvc_trace_stop()
    if st != zvc.ZVC_OK:
        raise zvc.ZvcError(st, "trace")
    return t


def measure_components(args, zvc, torch, xs, ns, C, dev, stream, peak):
    """Each kernel alone over the stack, and the offload / prefetch calls alone."""
    sh = stream.cuda_stream
    reps = max(10, min(args.steps, 50))
    outs = [torch.empty(zvc.zvc_size_bound(n, C), dtype=torch.uint8, device=dev) for n in ns]
    sizes = torch.zeros(len(ns), dtype=torch.int64, device=dev)
    wss = [zvc.new_workspace(zvc.zvc_workspace_size(n, C), dev) for n in ns]
    ys = [torch.empty_like(x) for x in xs]

    def comp():
        for l in range(len(ns)):
            zvc.zvc_compress(xs[l].data_ptr(), ns[l], C, outs[l].data_ptr(), outs[l].numel(),
                             sizes[l:l + 1].data_ptr(), wss[l].data_ptr(), wss[l].numel(), sh)

    comp()
    torch.cuda.synchronize(dev)
    S = [int(v) for v in sizes.cpu()]

    def decomp():
        for l in range(len(ns)):
            zvc.zvc_decompress(outs[l].data_ptr(), S[l], ys[l].data_ptr(), ns[l], C,
                               wss[l].data_ptr(), wss[l].numel(), sh)

    decomp()
    torch.cuda.synchronize(dev)
    for w in wss:
        if zvc.zvc_get_error(w.data_ptr(), sh) != zvc.ZVC_OK:
            raise RuntimeError("component run latched an error")
    N = sum(ns)
    tc = _trace(zvc, lambda: [comp() for _ in range(reps)])["compress"][1]
    td = _trace(zvc, lambda: [decomp() for _ in range(reps)])["decompress"][1]
    moved = 4 * N + sum(S)
    res = {"ratio": 4 * N / sum(S),
           "compress": {"gbs": reps * 4 * N / (tc / 1e3) / 1e9,
                        "hbm_gbs": reps * moved / (tc / 1e3) / 1e9,
                        "hbm_frac": reps * moved / (tc / 1e3) / 1e9 / peak},
           "decompress": {"gbs": reps * 4 * N / (td / 1e3) / 1e9,
                          "hbm_gbs": reps * moved / (td / 1e3) / 1e9,
                          "hbm_frac": reps * moved / (td / 1e3) / 1e9 / peak}}

    # the same stack through the batched calls: one compress launch and one decompress
    # launch over all five layers, so the ramp and drain of a launch are paid once
    bcap = zvc.zvc_batch_size_bound(ns, C)
    bout = torch.empty(bcap, dtype=torch.uint8, device=dev)
    bsize = torch.zeros(1, dtype=torch.int64, device=dev)
    bws = zvc.new_workspace(max(zvc.zvc_batch_workspace_size(ns, C), 256), dev)
    xptrs = [x.data_ptr() for x in xs]
    yptrs = [y.data_ptr() for y in ys]

    def bcomp():
        if zvc.zvc_compress_batched(xptrs, ns, C, bout.data_ptr(), bcap, bsize.data_ptr(),
                                    bws.data_ptr(), bws.numel(), sh) != zvc.ZVC_OK:
            raise RuntimeError("zvc_compress_batched")

    bcomp()
    torch.cuda.synchronize(dev)
    BS = int(bsize.item())

    def bdecomp():
        if zvc.zvc_decompress_batched(bout.data_ptr(), BS, yptrs, ns, C, bws.data_ptr(),
                                      bws.numel(), sh) != zvc.ZVC_OK:
            raise RuntimeError("zvc_decompress_batched")

    bdecomp()
    torch.cuda.synchronize(dev)
    if zvc.zvc_get_error(bws.data_ptr(), sh) != zvc.ZVC_OK or not all(
            torch.equal(x.view(torch.int32), y.view(torch.int32)) for x, y in zip(xs, ys)):
        raise RuntimeError("batched round trip failed")
    tbc = _trace(zvc, lambda: [bcomp() for _ in range(reps)])["compress"][1]
    tbd = _trace(zvc, lambda: [bdecomp() for _ in range(reps)])["decompress"][1]
    bmoved = 4 * N + BS
    for key, t in (("compress_batched", tbc), ("decompress_batched", tbd)):
        res[key] = {"gbs": reps * 4 * N / (t / 1e3) / 1e9,
                    "hbm_gbs": reps * bmoved / (t / 1e3) / 1e9,
                    "hbm_frac": reps * bmoved / (t / 1e3) / 1e9 / peak,
                    "launches_per_pass": 1}

    # offload alone and prefetch alone (wall time on the stream, events)
    hcap = [zvc.zvc_offload_host_bound(n, C) for n in ns]
    hb = [torch.empty(c, dtype=torch.uint8, pin_memory=True) for c in hcap]
    ows = [zvc.new_workspace(zvc.zvc_offload_workspace_size(n, C), dev) for n in ns]
    hs = [0] * len(ns)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    torch.cuda.synchronize(dev)
    ev[0].record(stream)
    for _ in range(reps):
        for l in range(len(ns)):
            _, hs[l] = zvc.zvc_offload(xs[l].data_ptr(), ns[l], C, hb[l].data_ptr(), hcap[l],
                                       ows[l].data_ptr(), ows[l].numel(), sh)
    zvc.zvc_offload_join(sh)  # the offload is done when its copies are
    ev[1].record(stream)
    for _ in range(reps):
        for l in range(len(ns)):
            zvc.zvc_prefetch(hb[l].data_ptr(), hs[l], ys[l].data_ptr(), ns[l], C,
                             ows[l].data_ptr(), ows[l].numel(), sh)
    ev[2].record(stream)
    torch.cuda.synchronize(dev)
    res["offload_gbs"] = reps * 4 * N / (ev[0].elapsed_time(ev[1]) / 1e3) / 1e9
    res["prefetch_gbs"] = reps * 4 * N / (ev[1].elapsed_time(ev[2]) / 1e3) / 1e9

    # plain uncompressed pinned copies of the same bytes, for comparison
    hx = [torch.empty(n, dtype=torch.float32, pin_memory=True) for n in ns]
    ev[0].record(stream)
    for _ in range(reps):
        for l in range(len(ns)):
            hx[l].copy_(xs[l].view(-1), non_blocking=True)
    ev[1].record(stream)
    for _ in range(reps):
        for l in range(len(ns)):
            ys[l].view(-1).copy_(hx[l], non_blocking=True)
    ev[2].record(stream)
    torch.cuda.synchronize(dev)
    res["plain_d2h_gbs"] = reps * 4 * N / (ev[0].elapsed_time(ev[1]) / 1e3) / 1e9
    res["plain_h2d_gbs"] = reps * 4 * N / (ev[1].elapsed_time(ev[2]) / 1e3) / 1e9
    return res


def run_profile_case(args):
    """Warm-up launches, then three timed groups of ten back-to-back launches of one kernel
    on AlexNet layer 0 (batch 128 x 96 x 55 x 55 fp32, 60% non-zero), or with
    --profile-density D on a flat map of as many words with a fraction D non-zero; prints
    the mean CUDA-event time per launch of each group."""
    import torch

    from activation_sparsity_compression_gb300 import build as zbuild
    zbuild.build()
    import activation_sparsity_compression_gb300 as zvc
    import workloads

    C = args.chunk_elems
    if args.profile.endswith("_batch"):
        return run_profile_batch(args, torch, zvc, workloads)
    g = torch.Generator(device="cuda").manual_seed(1)
    c, h, w, d = workloads.ALEXNET_LAYERS[0]
    if args.profile_layer:
        x = workloads.alexnet_stack(device="cuda")[args.profile_layer]
    elif args.profile_density is None:
        b = torch.tensor(workloads.alexnet_biases(c, d, 1), device="cuda").view(1, c, 1, 1)
        x = torch.relu_(torch.randn((128, c, h, w), generator=g, device="cuda").add_(b))
    else:
        x = workloads.density_sweep(args.profile_density, "iid", device="cuda",
                                    n=128 * c * h * w)[0]
    n = x.numel()
    out = torch.empty(zvc.zvc_size_bound(n, C), dtype=torch.uint8, device="cuda")
    size = torch.zeros(1, dtype=torch.int64, device="cuda")
    ws = zvc.new_workspace(zvc.zvc_workspace_size(n, C))
    y = torch.empty_like(x)
    sh = torch.cuda.current_stream().cuda_stream
    assert zvc.zvc_compress(x.data_ptr(), n, C, out.data_ptr(), out.numel(), size.data_ptr(),
                            ws.data_ptr(), ws.numel(), sh) == zvc.ZVC_OK
    S = int(size.item())
    if args.profile == "compress":
        def launch():
            zvc.zvc_compress(x.data_ptr(), n, C, out.data_ptr(), out.numel(), size.data_ptr(),
                             ws.data_ptr(), ws.numel(), sh)
    else:
        def launch():
            zvc.zvc_decompress(out.data_ptr(), S, y.data_ptr(), n, C, ws.data_ptr(), ws.numel(), sh)
    launch()
    # launches are queued back to back, so the device never waits for the host between
    # them; each entry is the mean over a group of `reps` launches
    reps = 10
    times = []
    for _ in range(4):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            launch()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) / reps)
    assert zvc.zvc_get_error(ws.data_ptr(), sh) == zvc.ZVC_OK
    if args.profile == "decompress":
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    moved = 4 * n + S
    print(json.dumps({"profile": args.profile, "density": args.profile_density,
                      "layer": args.profile_layer, "n": n,
                      "stream_bytes": S,
                      "ms": times[1:], "hbm_gbs": [moved / (t / 1e3) / 1e9 for t in times[1:]]}))
    return 0


def run_profile_batch(args, torch, zvc, workloads):
    """Launches of one batched kernel on the GoogLeNet batch at --profile-batch B: one
    compress launch to learn the stream size, one warm-up launch of the profiled kernel,
    then three timed groups of five back-to-back launches. The small case for ncu captures
    of the bench step's kernels (B = 16: 189 M words, 755 MB, larger than L2)."""
    C = args.chunk_elems
    xs = workloads.googlenet_batch(device="cuda", batch=args.profile_batch)
    ns = [x.numel() for x in xs]
    n = sum(ns)
    cap = zvc.zvc_batch_size_bound(ns, C)
    out = torch.empty(cap, dtype=torch.uint8, device="cuda")
    size = torch.zeros(1, dtype=torch.int64, device="cuda")
    ws = zvc.new_workspace(max(zvc.zvc_batch_workspace_size(ns, C), 256))
    ys = [torch.empty_like(x) for x in xs]
    xp, yp = [x.data_ptr() for x in xs], [y.data_ptr() for y in ys]
    sh = torch.cuda.current_stream().cuda_stream

    def bcomp():
        zvc.zvc_compress_batched(xp, ns, C, out.data_ptr(), cap, size.data_ptr(), ws.data_ptr(),
                                 ws.numel(), sh)
    bcomp()
    torch.cuda.synchronize()
    S = int(size.item())

    def bdecomp():
        zvc.zvc_decompress_batched(out.data_ptr(), S, yp, ns, C, ws.data_ptr(), ws.numel(), sh)
    launch = bcomp if args.profile == "compress_batch" else bdecomp
    best, times = _per_launch_ms(torch, launch, reps=5, groups=3)
    if args.profile == "decompress_batch" and not all(
            torch.equal(x.view(torch.int32), y.view(torch.int32)) for x, y in zip(xs, ys)):
        raise RuntimeError("batch round trip is not bit-exact")
    if zvc.zvc_get_error(ws.data_ptr(), sh) != zvc.ZVC_OK:
        raise RuntimeError("a device error was latched")
    moved = 4 * n + S
    print(json.dumps({"profile": args.profile, "batch": args.profile_batch, "n": n,
                      "stream_bytes": S, "ms": times,
                      "hbm_gbs": [moved / (t / 1e3) / 1e9 for t in times]}))
    return 0


def _per_launch_ms(torch, launch, reps=10, groups=3):
    """Mean CUDA-event time of one launch in each of `groups` groups of `reps` back-to-back
    launches on the current stream (after one warm-up launch); returns (best, all)."""
    launch()
    times = []
    for _ in range(groups):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            launch()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) / reps)
    return min(times), times


def _graph_per_launch_ms(torch, launch_on, reps=10, groups=3):
    """Per-launch time of `reps` launches captured in one CUDA graph (launch_on(stream)
    enqueues one launch on the given stream handle), best of `groups` replays."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(reps):
            launch_on(s.cuda_stream)
    g.replay()
    times = []
    for _ in range(groups):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) / reps)
    del g
    return min(times)


def run_configs(args):
    """Compress and decompress alone (device buffers, back-to-back launches) on each input
    configuration: the single 1x64x56x56 map (L2-resident: its GB/s is an L2 figure), each
    AlexNet layer, VGG conv1_2 at batch 64, the 2^28-word density sweep (9 densities, i.i.d.
    and 1024-word blocks), and the 57-tensor GoogLeNet batch through one batched launch each
    way. Every case is checked bit-exact after decompression. The single map and the
    AlexNet layers are also timed as 10 launches captured in a CUDA graph and replayed
    (graph_* keys), which removes most of the gap between back-to-back launches."""
    import torch

    from activation_sparsity_compression_gb300 import build as zbuild
    zbuild.build()
    import activation_sparsity_compression_gb300 as zvc
    import workloads

    C = args.chunk_elems
    peak, peak_kind = hbm_peak()
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    cases = []

    def ok(st, where):
        if st != zvc.ZVC_OK:
            raise zvc.ZvcError(st, where)

    def record(name, ns, S, tc, td, extra=None):
        n = sum(ns)
        moved = 4 * n + S
        c = {"case": name, "n_words": n, "stream_bytes": S, "ratio": 4 * n / S,
             "compress_us": tc * 1e3, "decompress_us": td * 1e3,
             "compress_gbs": 4 * n / (tc / 1e3) / 1e9,
             "decompress_gbs": 4 * n / (td / 1e3) / 1e9,
             "compress_hbm_frac": moved / (tc / 1e3) / 1e9 / peak,
             "decompress_hbm_frac": moved / (td / 1e3) / 1e9 / peak}
        if extra:
            c.update(extra)
        cases.append(c)
        print(json.dumps(c), file=sys.stderr, flush=True)

    def single(name, x, extra=None, graph=False):
        n = x.numel()
        cap = zvc.zvc_size_bound(n, C)
        out = torch.empty(cap, dtype=torch.uint8, device="cuda")
        size = torch.zeros(1, dtype=torch.int64, device="cuda")
        ws = zvc.new_workspace(zvc.zvc_workspace_size(n, C))
        y = torch.empty_like(x)

        def comp(s=sh):
            ok(zvc.zvc_compress(x.data_ptr(), n, C, out.data_ptr(), cap, size.data_ptr(),
                                ws.data_ptr(), ws.numel(), s), "zvc_compress")
        comp()
        torch.cuda.synchronize()
        S = int(size.item())

        def decomp(s=sh):
            ok(zvc.zvc_decompress(out.data_ptr(), S, y.data_ptr(), n, C, ws.data_ptr(),
                                  ws.numel(), s), "zvc_decompress")
        tc, _ = _per_launch_ms(torch, comp)
        td, _ = _per_launch_ms(torch, decomp)
        extra = dict(extra or {})
        if graph:
            moved = 4 * n + S
            gc = _graph_per_launch_ms(torch, comp)
            gd = _graph_per_launch_ms(torch, decomp)
            extra.update({"graph_compress_us": gc * 1e3, "graph_decompress_us": gd * 1e3,
                          "graph_compress_hbm_frac": moved / (gc / 1e3) / 1e9 / peak,
                          "graph_decompress_hbm_frac": moved / (gd / 1e3) / 1e9 / peak})
            torch.cuda.synchronize()
            if int(size.item()) != S:
                raise RuntimeError(f"{name}: a graph replay changed the stream size")
        if zvc.zvc_get_error(ws.data_ptr(), sh) != zvc.ZVC_OK or not torch.equal(
                x.view(torch.int32), y.view(torch.int32)):
            raise RuntimeError(f"{name}: round trip is not bit-exact")
        record(name, [n], S, tc, td, extra)
        del out, y, ws

    single("single_relu 1x64x56x56", workloads.single_relu(device="cuda")[0],
           {"note": "803 KB: L2-resident, so its GB/s are L2 figures"}, graph=True)
    for l, x in enumerate(workloads.alexnet_stack(device="cuda")):
        cc, hh, ww, d = workloads.ALEXNET_LAYERS[l]
        single(f"alexnet layer {l} 128x{cc}x{hh}x{ww} ({int(d * 100)}% non-zero)", x,
               graph=True)
    torch.cuda.empty_cache()
    single("vgg_conv12 64x64x224x224", workloads.vgg_conv12(device="cuda")[0])
    torch.cuda.empty_cache()
    for structure in ("iid", "block"):
        for d in workloads.SWEEP_DENSITIES:
            x = workloads.density_sweep(d, structure, device="cuda")[0]
            single(f"sweep 2^28 {structure} {d:.2f}", x, {"density": d, "structure": structure})
            del x
            torch.cuda.empty_cache()

    # the GoogLeNet batch: one batched launch each way over all 57 tensors
    xs = workloads.googlenet_batch(device="cuda")
    ns = [x.numel() for x in xs]
    cap = zvc.zvc_batch_size_bound(ns, C)
    out = torch.empty(cap, dtype=torch.uint8, device="cuda")
    size = torch.zeros(1, dtype=torch.int64, device="cuda")
    ws = zvc.new_workspace(max(zvc.zvc_batch_workspace_size(ns, C), 256))
    ys = [torch.empty_like(x) for x in xs]
    xp, yp = [x.data_ptr() for x in xs], [y.data_ptr() for y in ys]

    def bcomp():
        zvc.zvc_compress_batched(xp, ns, C, out.data_ptr(), cap, size.data_ptr(), ws.data_ptr(),
                                 ws.numel(), sh)
    bcomp()
    torch.cuda.synchronize()
    S = int(size.item())

    def bdecomp():
        zvc.zvc_decompress_batched(out.data_ptr(), S, yp, ns, C, ws.data_ptr(), ws.numel(), sh)
    tc, _ = _per_launch_ms(torch, bcomp, reps=3)
    td, _ = _per_launch_ms(torch, bdecomp, reps=3)
    if zvc.zvc_get_error(ws.data_ptr(), sh) != zvc.ZVC_OK or not all(
            torch.equal(x.view(torch.int32), y.view(torch.int32)) for x, y in zip(xs, ys)):
        raise RuntimeError("googlenet batch: round trip is not bit-exact")
    record("googlenet batch, 57 tensors, one batched launch each way", ns, S, tc, td,
           {"tensors": len(ns)})

    print(json.dumps({"metric": "ZVC compress/decompress per input configuration",
                      "unit": "GB/s (uncompressed) and fraction of HBM", "peak": peak,
                      "peak_kind": peak_kind, "chunk_elems": C, "data": "synthetic",
                      "timing": "CUDA events, one warm-up launch, best of 3 groups of "
                                "back-to-back launches (10, or 3 for the batch)",
                      "cases": cases}), flush=True)
    return 0


def run_configs16(args):
    """The 16-bit calls alone (device buffers, back-to-back launches) on bf16 copies of the
    single-tensor configurations: each AlexNet layer, VGG conv1_2 at batch 64, and the
    2^28-word density sweep (i.i.d. and 1024-word blocks). Algorithmic bytes are 2n + S.
    Every case is checked bit-exact after decompression."""
    import torch

    from activation_sparsity_compression_gb300 import build as zbuild
    zbuild.build()
    import activation_sparsity_compression_gb300 as zvc
    import workloads

    C = args.chunk_elems
    peak, peak_kind = hbm_peak()
    sh = torch.cuda.current_stream().cuda_stream
    cases = []

    def single(name, x32, extra=None):
        x = x32.to(torch.bfloat16).contiguous().view(-1)
        del x32
        n = x.numel()
        cap = zvc.zvc_size_bound16(n, C)
        out = torch.empty(cap, dtype=torch.uint8, device="cuda")
        size = torch.zeros(1, dtype=torch.int64, device="cuda")
        ws = zvc.new_workspace(zvc.zvc_workspace_size(n, C))
        y = torch.empty_like(x)

        def comp():
            zvc.zvc_compress16(x.data_ptr(), n, C, out.data_ptr(), cap, size.data_ptr(),
                               ws.data_ptr(), ws.numel(), sh)
        comp()
        torch.cuda.synchronize()
        S = int(size.item())

        def decomp():
            zvc.zvc_decompress16(out.data_ptr(), S, y.data_ptr(), n, C, ws.data_ptr(),
                                 ws.numel(), sh)
        tc, _ = _per_launch_ms(torch, comp)
        td, _ = _per_launch_ms(torch, decomp)
        if zvc.zvc_get_error(ws.data_ptr(), sh) != zvc.ZVC_OK or not torch.equal(
                x.view(torch.int16), y.view(torch.int16)):
            raise RuntimeError(f"{name}: 16-bit round trip is not bit-exact")
        moved = 2 * n + S
        c = {"case": name, "n_words": n, "stream_bytes": S, "ratio": 2 * n / S,
             "compress_us": tc * 1e3, "decompress_us": td * 1e3,
             "compress_gbs": 2 * n / (tc / 1e3) / 1e9, "decompress_gbs": 2 * n / (td / 1e3) / 1e9,
             "compress_hbm_frac": moved / (tc / 1e3) / 1e9 / peak,
             "decompress_hbm_frac": moved / (td / 1e3) / 1e9 / peak}
        if extra:
            c.update(extra)
        cases.append(c)
        print(json.dumps(c), file=sys.stderr, flush=True)
        del out, y, ws, x

    for l, x in enumerate(workloads.alexnet_stack(device="cuda")):
        cc, hh, ww, d = workloads.ALEXNET_LAYERS[l]
        single(f"alexnet layer {l} 128x{cc}x{hh}x{ww} ({int(d * 100)}% non-zero), bf16", x)
    torch.cuda.empty_cache()
    single("vgg_conv12 64x64x224x224, bf16", workloads.vgg_conv12(device="cuda")[0])
    torch.cuda.empty_cache()
    for structure in ("iid", "block"):
        for d in workloads.SWEEP_DENSITIES:
            x = workloads.density_sweep(d, structure, device="cuda")[0]
            single(f"sweep 2^28 {structure} {d:.2f}, bf16", x, {"density": d, "structure": structure})
            del x
            torch.cuda.empty_cache()
    print(json.dumps({"metric": "ZVC on 16-bit words, compress/decompress per configuration",
                      "unit": "GB/s (uncompressed) and fraction of HBM", "peak": peak,
                      "peak_kind": peak_kind, "chunk_elems": C, "word_bytes": 2,
                      "data": "synthetic (bf16 copies of the fp32 configurations)",
                      "timing": "CUDA events, one warm-up launch, best of 3 groups of 10 "
                                "back-to-back launches",
                      "cases": cases}), flush=True)
    return 0


# ------------------------------------------------------------------ training step with offload
TRAIN_MODEL = ("deep CNN: conv 3->128 (3x3, stride 2) + ReLU, then 12 x (conv 128->128 3x3 + "
               "ReLU) at 112x112, global average pool, linear 128->1000; batch 64, 3x224x224, "
               "random weights and inputs")


def _deep_cnn():
    import torch
    nn = torch.nn
    torch.manual_seed(0)
    layers = [nn.Conv2d(3, 128, 3, stride=2, padding=1), nn.ReLU()]
    for _ in range(12):
        layers += [nn.Conv2d(128, 128, 3, padding=1), nn.ReLU()]
    layers += [nn.AdaptiveAvgPool2d(1), nn.Flatten(), nn.Linear(128, 1000)]
    return nn.Sequential(*layers).cuda()


def run_train(args):
    """The path inside a training step (the vDNN setting of section V.D): forward and
    backward of a CNN whose saved activations are (a) kept in HBM, (b) compressed and
    offloaded to pinned host memory during forward and prefetched back during backward, or
    (c) kept compressed in HBM. Reports time per step, peak device memory and the
    compression of the saved activations; the gradients of (b) and (c) must equal (a)'s
    bit for bit."""
    import torch

    from activation_sparsity_compression_gb300 import build as zbuild
    zbuild.build()
    from activation_sparsity_compression_gb300.offload import ActivationOffload

    torch.backends.cudnn.deterministic = True
    torch.backends.cudnn.benchmark = False
    model = _deep_cnn()
    g = torch.Generator(device="cuda").manual_seed(1)
    x = torch.randn(64, 3, 224, 224, device="cuda", generator=g)

    def step(off):
        model.zero_grad(set_to_none=True)
        if off is None:
            loss = model(x).square().mean()
        else:
            with off:
                loss = model(x).square().mean()
        loss.backward()

    res, grads = {}, {}
    steps = max(3, min(args.steps, 20))
    for mode in ("keep", "host", "device"):
        off = None if mode == "keep" else ActivationOffload(where=mode)
        for _ in range(max(args.warmup, 2)):
            step(off)
        torch.cuda.synchronize()
        torch.cuda.reset_peak_memory_stats()
        base = torch.cuda.memory_allocated()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            step(off)
        e1.record()
        torch.cuda.synchronize()
        if off is not None:
            off.check_errors()
        grads[mode] = [p.grad.clone() for p in model.parameters()]
        r = {"ms_per_step": e0.elapsed_time(e1) / steps,
             "peak_extra_gb": (torch.cuda.max_memory_allocated() - base) / 1e9}
        if off is not None:
            st = off.stats
            passes = max(args.warmup, 2) + steps
            r["compressed_gb_in_per_step"] = st["bytes_in"] / passes / 1e9
            r["compressed_gb_out_per_step"] = st["bytes_stored"] / passes / 1e9
            r["ratio"] = st["bytes_in"] / max(st["bytes_stored"], 1)
        res[mode] = r
    identical = all(torch.equal(a, b) for m in ("host", "device")
                    for a, b in zip(grads["keep"], grads[m]))
    line = {"metric": "training step with ZVC activation offload", "unit": "ms",
            "higher_is_better": False, "config": {"model": TRAIN_MODEL},
            "data": "synthetic", "gradients_bit_identical": identical, "modes": res}
    print(json.dumps(line), flush=True)
    return 0 if identical else 1


# ------------------------------------------------------------------ layouts: ZVC against RLE
def run_layouts(args):
    """Compression ratio (4n / stream bytes) of ZVC and of RLE for the same activations in
    three layouts (Rhu et al., section VII.A: ZVC's ratio does not depend on the layout,
    RLE's does), computed by this library's kernels, plus back-to-back kernel times of RLE
    next to ZVC on AlexNet layer 0."""
    import torch

    from activation_sparsity_compression_gb300 import build as zbuild
    zbuild.build()
    import activation_sparsity_compression_gb300 as zvc
    import workloads

    C, W = args.chunk_elems, 1024
    dev = torch.device("cuda", 0)
    sh = torch.cuda.current_stream(dev).cuda_stream

    def sizes(x):
        n = x.numel()
        out = torch.empty(max(zvc.zvc_size_bound(n, C), zvc.zvc_rle_size_bound(n, W)),
                          dtype=torch.uint8, device=dev)
        size = torch.zeros(2, dtype=torch.int64, device=dev)
        ws = zvc.new_workspace(max(zvc.zvc_workspace_size(n, C), zvc.zvc_rle_workspace_size(n, W)),
                               dev)
        assert zvc.zvc_compress(x.data_ptr(), n, C, out.data_ptr(), out.numel(), size.data_ptr(),
                                ws.data_ptr(), ws.numel(), sh) == zvc.ZVC_OK
        assert zvc.zvc_rle_compress(x.data_ptr(), n, W, out.data_ptr(), out.numel(),
                                    size.data_ptr() + 8, ws.data_ptr(), ws.numel(), sh) == zvc.ZVC_OK
        assert zvc.zvc_get_error(ws.data_ptr(), sh) == zvc.ZVC_OK
        s_zvc, s_rle = (int(v) for v in size.tolist())
        return 4 * n / s_zvc, 4 * n / s_rle

    layouts = {"NCHW": lambda t: t, "NHWC": lambda t: t.permute(0, 2, 3, 1),
               "CHWN": lambda t: t.permute(1, 2, 3, 0)}
    res = {}
    cases = [("alexnet_stack", workloads.alexnet_stack(device=dev)),
             ("vgg_conv12", workloads.vgg_conv12(device=dev))]
    for name, xs in cases:
        res[name] = {}
        for lname, f in layouts.items():
            tot_in = tot_zvc = tot_rle = 0.0
            for x in xs:
                t = f(x).contiguous()
                rz, rr = sizes(t)
                tot_in += 4 * t.numel()
                tot_zvc += 4 * t.numel() / rz
                tot_rle += 4 * t.numel() / rr
                del t
            res[name][lname] = {"zvc_ratio": tot_in / tot_zvc, "rle_ratio": tot_in / tot_rle}
        del xs
        torch.cuda.empty_cache()

    # kernel times on AlexNet layer 0 (back-to-back launches, CUDA events)
    x = workloads.alexnet_stack(device=dev)[0]
    n = x.numel()
    times = {}
    for codec in ("zvc", "rle"):
        cap = zvc.zvc_size_bound(n, C) if codec == "zvc" else zvc.zvc_rle_size_bound(n, W)
        out = torch.empty(cap, dtype=torch.uint8, device=dev)
        size = torch.zeros(1, dtype=torch.int64, device=dev)
        wsb = zvc.zvc_workspace_size(n, C) if codec == "zvc" else zvc.zvc_rle_workspace_size(n, W)
        ws = zvc.new_workspace(wsb, dev)
        y = torch.empty_like(x)

        def comp():
            if codec == "zvc":
                return zvc.zvc_compress(x.data_ptr(), n, C, out.data_ptr(), cap, size.data_ptr(),
                                        ws.data_ptr(), ws.numel(), sh)
            return zvc.zvc_rle_compress(x.data_ptr(), n, W, out.data_ptr(), cap, size.data_ptr(),
                                        ws.data_ptr(), ws.numel(), sh)
        assert comp() == zvc.ZVC_OK
        S = int(size.item())

        def decomp():
            if codec == "zvc":
                return zvc.zvc_decompress(out.data_ptr(), S, y.data_ptr(), n, C, ws.data_ptr(),
                                          ws.numel(), sh)
            return zvc.zvc_rle_decompress(out.data_ptr(), S, y.data_ptr(), n, W, ws.data_ptr(),
                                          ws.numel(), sh)
        r = {}
        for nm, fn in (("compress", comp), ("decompress", decomp)):
            fn()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(10):
                fn()
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / 10
            r[nm] = {"ms": ms, "gbs_uncompressed": 4 * n / (ms / 1e3) / 1e9}
        assert zvc.zvc_get_error(ws.data_ptr(), sh) == zvc.ZVC_OK
        assert torch.equal(y.view(torch.int32), x.view(torch.int32))
        r["ratio"] = 4 * n / S
        times[codec] = r
    line = {"metric": "compression ratio by layout, ZVC vs RLE (4 KB RLE windows)",
            "unit": "x", "higher_is_better": True, "data": "synthetic",
            "config": {"zvc_chunk_elems": C, "rle_window": W,
                       "workloads": ["alexnet_stack batch 128", "vgg_conv12 batch 64"]},
            "ratios": res, "alexnet_layer0_kernels": times}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.write_traffic:
        return write_traffic(args.write_traffic, args.chunk_elems, args.profile_batch)
    if args.configs:
        return run_configs(args)
    if args.configs16:
        return run_configs16(args)
    if args.train:
        return run_train(args)
    if args.layouts:
        return run_layouts(args)
    if args.profile:
        return run_profile_case(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
