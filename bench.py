#!/usr/bin/env python3
"""Benchmark of the ZVC hot path on the AlexNet-shaped activation stack.

One step is the whole path on the 5 conv activations of batch 128 (83,210,240 fp32 words,
333 MB): every layer is offloaded (compressed on the GPU, compressed bytes copied to
pinned host memory) and then prefetched in reverse layer order (copied back and
decompressed), as vDNN offloads activations in forward and prefetches them for backward
propagation (Rhu et al., "Compressing DMA Engine", section V.D). `value` is uncompressed
GB/s through that round trip with the activations already in HBM.

The same line reports, measured in the same run:
  roofline      the dominant kernel's algorithmic bytes (4n read + S written for
                compress, S read + 4n written for decompress) per device second, against
                the measured HBM copy bandwidth; `kernels` lists every traced kernel's
                launches, device time and share of the step
  compress / decompress   each kernel alone over the stack (device buffers)
  e2e           the step with inputs in pinned host memory: H2D of the inputs and D2H of
                the restored activations inside the timed region
  cpu_baseline  the single-threaded CPU oracle on a bounded sample of the same workload
`--impl reference` times that oracle alone (the pages describe hardware; the oracle is
the only other implementation of this path).
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "ZVC compress/decompress GB/s (uncompressed) and % of HBM roofline; ratio"
WORKLOAD = ("alexnet_stack: batch-128 AlexNet conv activations 96x55x55, 256x27x27, "
            "384x13x13, 384x13x13, 256x13x13 fp32 = ReLU(x + b_c), non-zero 60/45/35/30/20%")
FALLBACK_HBM_GBS = 6800.0


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--chunk-elems", type=int, default=4096)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--profile", choices=["compress", "decompress"],
                   help="run a few launches of one kernel on AlexNet layer 0 (149 MB) and "
                        "exit: the small case for ncu captures")
    p.add_argument("--profile-density", type=float, default=None, metavar="D",
                   help="with --profile: a flat map of the same size with a fraction D of "
                        "i.i.d. non-zero words, instead of AlexNet layer 0")
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
    p.add_argument("--write-traffic", nargs=2, metavar=("COMPRESS_CSV", "DECOMPRESS_CSV"),
                   help="turn ncu DRAM counters of one step's launches (see TRAFFIC_FILE) "
                        "into that file, keyed by the kernels' source hashes, and exit")
    return p.parse_args(argv)


# ------------------------------------------------------------------ DRAM traffic record
# `traffic` in the bench line comes from ncu counters taken on this very step: the
# dram__bytes_read.sum + dram__bytes_write.sum of every compress (decompress) launch of
# one timed step, captured with
#   ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum
#       --clock-control none -k regex:^<kernel> -s <L> -c <L> --csv --log-file <csv>
#       python bench.py --steps 2 --warmup 1 --no-cpu-baseline
# with L the kernel's launches per step (one per offload segment: 6 for the AlexNet stack),
# so that the warm-up step's launches are skipped and the next step's captured: together
# they cover every word of the stack once. The record holds bytes per word and the hash of the
# kernel's sources; once a source changes the record no longer applies and `traffic` is
# null until it is captured again.
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


def ncu_dram_bytes(csv_path: str):
    """Per-launch dram__bytes_read.sum + dram__bytes_write.sum from an ncu --csv log."""
    import csv
    rows = list(csv.reader(open(csv_path)))
    h = next(i for i, r in enumerate(rows) if r and r[0] == "ID")
    hdr = rows[h]
    ii, mi, vi, ui = (hdr.index(x) for x in ("ID", "Metric Name", "Metric Value", "Metric Unit"))
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    per = {}
    for r in rows[h + 1:]:
        if len(r) > vi and r[mi] in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            per[r[ii]] = per.get(r[ii], 0.0) + float(r[vi].replace(",", "")) * scale[r[ui]]
    return [per[k] for k in sorted(per, key=int)]


def launches_per_step(chunk_elems: int) -> int:
    """Compress (and decompress) launches of one bench step: one per offload segment."""
    import activation_sparsity_compression_gb300 as zvc
    import workloads
    ns = [c * h * w * 128 for c, h, w, _ in workloads.ALEXNET_LAYERS]
    return sum(-(-n // zvc.zvc_offload_segment_elems(n, chunk_elems)) for n in ns)


def write_traffic(csvs, chunk_elems):
    import workloads
    n_words = sum(c * h * w * 128 for c, h, w, _ in workloads.ALEXNET_LAYERS)
    L = launches_per_step(chunk_elems)
    rec = {"command": "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,"
                      f"gpu__time_duration.sum --clock-control none -k regex:^<kernel> -s {L} "
                      f"-c {L} --csv --log-file <csv> python bench.py --steps 2 --warmup 1 "
                      "--no-cpu-baseline",
           "words_per_step": n_words, "kernels": {}}
    for kernel, path in zip(("compress_kernel", "decompress_kernel"), csvs):
        b = ncu_dram_bytes(path)
        if len(b) != L:
            raise SystemExit(f"{path}: {len(b)} launches captured, one step has {L}")
        rec["kernels"][kernel] = {"source_sha256": kernel_source_hash(kernel), "launches": len(b),
                                  "dram_bytes": sum(b), "dram_bytes_per_word": sum(b) / n_words}
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


# ------------------------------------------------------------------ CPU oracle leg
def oracle_round_trip(batch: int, chunk_elems: int, budget_s: float):
    """Times the CPU oracle (encode then decode, i.e. compress -> host -> decompress) on
    the stack generated at a reduced batch, passing over it repeatedly until budget_s of
    CPU work is done (at least one whole pass). Returns (GB/s, words, seconds, passes)."""
    import numpy as np

    import oracle
    import workloads

    lib = oracle.load()
    layers = [x.numpy().view(np.uint32).reshape(-1) for x in
              workloads.alexnet_stack(device="cpu", batch=batch)]
    done = passes = 0
    t0 = time.perf_counter()
    while True:
        for w in layers:
            s = oracle.encode(w, chunk_elems, lib=lib)
            st, back = oracle.decode(s, w.size, chunk_elems, lib=lib)
            if st != oracle.OK or (passes == 0 and not np.array_equal(back, w)):
                raise RuntimeError("oracle round trip failed")
            done += w.size
        passes += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return 4 * done / dt / 1e9, done, dt, passes


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import numpy as np

    import oracle
    import workloads

    lib = oracle.load()
    batch = 16  # 1/8 of the batch-128 stack per step: 10.4 M words, about 0.1 s
    layers = [x.numpy().view(np.uint32).reshape(-1) for x in
              workloads.alexnet_stack(device="cpu", batch=batch)]
    n = sum(w.size for w in layers)

    def step():
        for w in layers:
            s = oracle.encode(w, args.chunk_elems, lib=lib)
            st, _ = oracle.decode(s, w.size, args.chunk_elems, lib=lib)
            if st != oracle.OK:
                raise RuntimeError("oracle decode failed")

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = 4 * n * args.steps / dt / 1e9
    sample = (f"alexnet_stack at batch {batch} (1/8 of batch 128, {n} words) per step; "
              "oracle encode + decode, single thread")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "chunk_elems": args.chunk_elems,
                       "sample_batch": batch},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU leg
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
    xs = workloads.alexnet_stack(device=dev, seed=1 + 100 * rank)
    ns = [x.numel() for x in xs]
    N = sum(ns)
    L = len(xs)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    def ok(st, where):
        if st != zvc.ZVC_OK:
            raise zvc.ZvcError(st, where)

    hcap = [zvc.zvc_offload_host_bound(n, C) for n in ns]
    hbuf = [torch.empty(c, dtype=torch.uint8, pin_memory=True) for c in hcap]
    ws = [zvc.new_workspace(zvc.zvc_offload_workspace_size(n, C), dev) for n in ns]
    ys = [torch.empty_like(x) for x in xs]
    hsize = [0] * L

    def step(inputs=xs, outputs=ys):
        for l in range(L):
            st, hsize[l] = zvc.zvc_offload(inputs[l].data_ptr(), ns[l], C, hbuf[l].data_ptr(),
                                           hcap[l], ws[l].data_ptr(), ws[l].numel(), sh)
            ok(st, "zvc_offload")
        for l in reversed(range(L)):
            ok(zvc.zvc_prefetch(hbuf[l].data_ptr(), hsize[l], outputs[l].data_ptr(), ns[l], C,
                                ws[l].data_ptr(), ws[l].numel(), sh), "zvc_prefetch")

    for _ in range(max(args.warmup, 1)):
        step()
    torch.cuda.synchronize(dev)
    for l in range(L):
        ok(zvc.zvc_get_error(ws[l].data_ptr(), sh), "device")
        if not torch.equal(xs[l].view(torch.int32), ys[l].view(torch.int32)):
            raise RuntimeError(f"round trip of layer {l} is not bit-exact")

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    sampler.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    ok(zvc.zvc_trace_start(), "trace")
    w0 = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    w1 = time.time()
    barrier()
    st, trace = zvc.zvc_trace_stop()
    ok(st, "trace")
    clocks = sampler.stop(w0, w1)
    ms = e0.elapsed_time(e1)
    max_ms = reduce_max(ms, dev)
    value = whole_job_gbs(4 * N, world, args.steps, max_ms)

    # bytes behind the dominant kernel, from the host copies' batch tables
    prefixes = [16 + 8 * (-(-n // zvc.zvc_offload_segment_elems(n, C)) + 1) for n in ns]
    seg_stream_bytes = sum(h - p for h, p in zip(hsize, prefixes))
    algo_bytes = args.steps * (4 * N + seg_stream_bytes)
    peak, peak_kind = hbm_peak()
    kern = max(trace, key=lambda k: trace[k][1])
    launches, kms = trace[kern]
    achieved = algo_bytes / (kms / 1e3) / 1e9
    per_launch_words = args.steps * N / launches
    traffic = traffic_per_launch(f"{kern}_kernel", per_launch_words)
    roofline = {"bound": "hbm", "kernel": f"{kern}_kernel", "achieved": achieved, "peak": peak,
                "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                "traffic": traffic, "traffic_unit": "bytes per launch",
                "algorithmic_bytes_per_launch": algo_bytes / launches,
                "avg_launch_us": kms / launches * 1e3, "share_of_step": kms / ms,
                # every traced kernel, for comparison with the ncu launch list's shares
                "kernels": {f"{k}_kernel": {"launches": v[0], "ms": v[1],
                                            "share_of_step": v[1] / ms}
                            for k, v in trace.items()}}

    extra = measure_components(args, zvc, torch, xs, ns, C, dev, stream, peak)
    e2e = measure_e2e(args, zvc, torch, xs, ns, C, dev, stream, step, hsize)

    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": max_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "n_words": N, "chunk_elems": C,
                       "step": "zvc_offload of 5 layers, then zvc_prefetch in reverse order",
                       "l2": "inputs larger than L2 (333 MB per step), no flush"},
            "ratio": extra.pop("ratio"),
            "link_bytes_per_step": sum(hsize),
            "roofline": roofline,
            "gpu_launches": trace["compress"][0] + trace["decompress"][0],
            "clocks": clocks, "e2e": e2e}
    line.update(extra)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        gbs, words, secs, passes = oracle_round_trip(batch=16, chunk_elems=C, budget_s=12.0)
        line["cpu_baseline"] = {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                "sample": f"alexnet_stack at batch 16 (1/8 of batch 128), "
                                          f"{passes} passes: {words} words encoded and "
                                          f"decoded in {secs:.1f} s, single thread"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


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


def measure_e2e(args, zvc, torch, xs, ns, C, dev, stream, step, hsize):
    """The step through the same C-ABI calls with the activations in pinned host memory:
    H2D of the inputs, offload, prefetch, D2H of the restored activations."""
    hx = [torch.empty(n, dtype=torch.float32, pin_memory=True) for n in ns]
    hy = [torch.empty(n, dtype=torch.float32, pin_memory=True) for n in ns]
    for h, x in zip(hx, xs):
        h.copy_(x.view(-1))
    dx = [torch.empty_like(x).view(-1) for x in xs]
    dy = [torch.empty_like(x).view(-1) for x in xs]

    def e2e_step():
        for d, h in zip(dx, hx):
            d.copy_(h, non_blocking=True)
        step(dx, dy)
        for h, d in zip(hy, dy):
            h.copy_(d, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    for h, x in zip(hy, hx):
        if not torch.equal(h.view(torch.int32), x.view(torch.int32)):
            raise RuntimeError("e2e round trip is not bit-exact")
    reps = max(5, min(args.steps, 50))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(reps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    max_ms = reduce_max(e0.elapsed_time(e1), dev)
    _, world, _ = dist_env()
    N = sum(ns)
    return {"value": whole_job_gbs(4 * N, world, reps, max_ms), "unit": "GB/s",
            "h2d_bytes_per_step": 4 * N + sum(hsize), "d2h_bytes_per_step": sum(hsize) + 4 * N,
            "steps": reps}


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
    g = torch.Generator(device="cuda").manual_seed(1)
    c, h, w, d = workloads.ALEXNET_LAYERS[0]
    if args.profile_density is None:
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
    print(json.dumps({"profile": args.profile, "density": args.profile_density, "n": n,
                      "stream_bytes": S,
                      "ms": times[1:], "hbm_gbs": [moved / (t / 1e3) / 1e9 for t in times[1:]]}))
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


def run_configs(args):
    """Compress and decompress alone (device buffers, back-to-back launches) on each input
    configuration: the single 1x64x56x56 map (L2-resident: its GB/s is an L2 figure), each
    AlexNet layer, VGG conv1_2 at batch 64, the 2^28-word density sweep (9 densities, i.i.d.
    and 1024-word blocks), and the 57-tensor GoogLeNet batch through one batched launch each
    way. Every case is checked bit-exact after decompression."""
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

    def single(name, x, extra=None):
        n = x.numel()
        cap = zvc.zvc_size_bound(n, C)
        out = torch.empty(cap, dtype=torch.uint8, device="cuda")
        size = torch.zeros(1, dtype=torch.int64, device="cuda")
        ws = zvc.new_workspace(zvc.zvc_workspace_size(n, C))
        y = torch.empty_like(x)

        def comp():
            zvc.zvc_compress(x.data_ptr(), n, C, out.data_ptr(), cap, size.data_ptr(),
                             ws.data_ptr(), ws.numel(), sh)
        comp()
        torch.cuda.synchronize()
        S = int(size.item())

        def decomp():
            zvc.zvc_decompress(out.data_ptr(), S, y.data_ptr(), n, C, ws.data_ptr(), ws.numel(), sh)
        tc, _ = _per_launch_ms(torch, comp)
        td, _ = _per_launch_ms(torch, decomp)
        if zvc.zvc_get_error(ws.data_ptr(), sh) != zvc.ZVC_OK or not torch.equal(
                x.view(torch.int32), y.view(torch.int32)):
            raise RuntimeError(f"{name}: round trip is not bit-exact")
        record(name, [n], S, tc, td, extra)
        del out, y, ws

    single("single_relu 1x64x56x56", workloads.single_relu(device="cuda")[0],
           {"note": "803 KB: L2-resident, so its GB/s are L2 figures"})
    for l, x in enumerate(workloads.alexnet_stack(device="cuda")):
        cc, hh, ww, d = workloads.ALEXNET_LAYERS[l]
        single(f"alexnet layer {l} 128x{cc}x{hh}x{ww} ({int(d * 100)}% non-zero)", x)
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
        return write_traffic(args.write_traffic, args.chunk_elems)
    if args.configs:
        return run_configs(args)
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
