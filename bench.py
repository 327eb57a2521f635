#!/usr/bin/env python
"""Benchmark of the Four Over Six NVFP4 hot path on B300.

Headline: NVFP4 4/6 quantization throughput (Gelem/s, and the HBM GB/s of the
quantize kernel against the measured copy bandwidth) on the weight set of one
Qwen3-8B decoder layer (q, k, v, o, gate, up, down: 192.9M bf16 values,
Student-t nu = 4, std 0.02), 1D 16-value blocks, round-to-nearest-even.  One
step quantizes all seven matrices through the public C-ABI call (the amax
pass and the quantize pass).  The step's inputs (386 MB) are larger than the
126 MB L2, so every matrix is evicted before it is read again.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fos|reference]

Under torchrun (N > 1) every rank quantizes its own copy of the weight set
(weak scaling, no data-path collective); the timing takes the max over ranks.
`--impl reference` times the CPU oracle (test infrastructure) on a bounded
sample of the same workload, on the host cores, on rank 0 only.

Secondary measurements (same JSON line): the activation (RHT, row-major and
transposed), gradient (stochastic rounding, 1D and 2D) and linear-layer
(quantize + NVFP4 GEMM) workloads, and an end-to-end number with host
buffers.  `--case NAME` runs one small case for profiling instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "NVFP4 4/6 quantize Gelem/s + HBM GB/s (% of peak); NVFP4 GEMM TFLOP/s"
WORKLOAD = ("qwen3-8b layer weights q,k,v,o,gate,up,down (192.9M bf16 values, Student-t nu=4 std 0.02); "
            "NVFP4 4/6, 1D 16-value blocks, RNE, swizzled 128x4 scales")
BYTES_PER_ELEM_QUANT = 2.0 + 0.5 + 1.0 / 16.0  # read bf16, write 4-bit code + 1/16 E4M3 scale
CPU_SAMPLE_ROWS = 2048  # rows of each matrix timed on the host for the CPU baseline
REF_SAMPLE_ROWS = 256  # rows of each matrix per step of the reference arm
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "quant_batch_step_traffic.txt")


def peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


def kernel_source_hash() -> str:
    """Hash of the code of the quantize kernels, comments and blank lines left
    out (to tell whether a recorded DRAM-traffic figure still belongs to the
    current kernels)."""
    import hashlib
    import re

    h = hashlib.sha256()
    for f in ("fos_quant.cu", "fos_device.cuh"):
        with open(os.path.join(ROOT, "adaptive_quantization_fos_b300", "csrc", f), encoding="utf-8") as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        code = [re.sub(r"//.*$", "", line).rstrip() for line in src.splitlines()]
        h.update("\n".join(line for line in code if line).encode())
    return h.hexdigest()[:16]


def recorded_traffic_per_elem() -> float | None:
    """DRAM bytes per value of the quantize kernel from the committed ncu
    summary, or None when it was taken on other kernel sources."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    kv = {}
    with open(TRAFFIC_FILE) as f:
        for line in f:
            if "=" in line and not line.startswith("#"):
                k, v = line.strip().split("=", 1)
                kv[k.strip()] = v.strip()
    if kv.get("source_sha") != kernel_source_hash():
        return None
    try:
        return float(kv["dram_bytes_per_value"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------- clocks


class ClockSampler:
    """Samples the SM clock and the clock-event reasons through NVML (the
    driver's libnvidia-ml, via ctypes) while the timed region runs."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
               0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}
    NVML_CLOCK_SM = 1

    def __init__(self, device_index: int, period_s: float = 0.001):
        import ctypes

        self.period = period_s
        self.samples: list[tuple[int, int]] = []
        self.times: list[float] = []
        self.window: tuple[float, float] | None = None
        self.max_mhz = None
        self._stop = threading.Event()
        self._ok = False
        self.err = ""
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise RuntimeError("nvmlInit failed")
            self.nv = nv
            self.h = ctypes.c_void_p()
            if not self._handle_by_bus(device_index) and nv.nvmlDeviceGetHandleByIndex_v2(
                    self._nvml_index(device_index), ctypes.byref(self.h)) != 0:
                raise RuntimeError("no NVML handle")
            v = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(self.h, self.NVML_CLOCK_SM, ctypes.byref(v)) == 0:
                self.max_mhz = v.value
            self._reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self._ok = True
        except Exception as e:  # noqa: BLE001
            self.err = str(e)

    def _handle_by_bus(self, idx) -> bool:
        import ctypes

        try:
            import torch

            pr = torch.cuda.get_device_properties(idx)
            bus = "%08X:%02X:%02X.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
            return self.nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.h)) == 0
        except Exception:  # noqa: BLE001
            return False

    @staticmethod
    def _nvml_index(idx: int) -> int:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        parts = [p for p in vis.split(",") if p.strip()]
        if idx < len(parts) and parts[idx].strip().isdigit():
            return int(parts[idx])
        return idx

    def _run(self):
        import ctypes

        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self.nv.nvmlDeviceGetClockInfo(self.h, self.NVML_CLOCK_SM, ctypes.byref(clk)) == 0 and \
                    self._reasons_fn(self.h, ctypes.byref(rs)) == 0:
                self.samples.append((clk.value, rs.value))
                self.times.append(time.perf_counter())
            time.sleep(self.period)

    def mark(self, t0: float, t1: float) -> None:
        """Host-time bounds of the timed region (the rest of the sampled
        window runs the same work untimed, so short regions get samples)."""
        self.window = (t0, t1)

    def __enter__(self):
        if self._ok:
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()
        return self

    def __exit__(self, *a):
        if self._ok:
            self._stop.set()
            self.t.join()

    def summary(self) -> dict:
        if not self._ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "note": self.err or "no samples"}
        bits = 0
        for _, r in self.samples:
            bits |= r
        out = {"sm_mhz": statistics.median(s for s, _ in self.samples), "sm_max_mhz": self.max_mhz,
               "reasons": [n for b, n in self.REASONS.items() if bits & b and n != "gpu_idle"],
               "samples": len(self.samples), "period_ms": self.period * 1e3}
        if self.window:
            inside = [s for (s, _), t in zip(self.samples, self.times) if self.window[0] <= t <= self.window[1]]
            out["samples_timed_region"] = len(inside)
            if inside:
                out["sm_mhz_timed_region"] = statistics.median(inside)
            out["note"] = ("sampled over the timed region and an untimed continuation of the same steps "
                           "(at least 0.3 s of load in all)")
        return out


# ------------------------------------------------------------ distributed


class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend: str):
        if self.world > 1:
            import torch.distributed as dist

            kw = {}
            if backend == "nccl":
                import torch

                kw["device_id"] = torch.device("cuda", self.local_rank)
            dist.init_process_group(backend, **kw)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v: float, device) -> float:
        if not self.pg:
            return v
        import torch

        t = torch.tensor([v], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ------------------------------------------------------------ CPU oracle


def host_cpu() -> dict:
    """The host's logical core count and CPU model (from /proc/cpuinfo)."""
    model = "unknown"
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    return {"nproc": n, "model": model}


def oracle_quantize_threads(orc, bits: np.ndarray, threads: int, pool) -> None:
    """The oracle's quantization of one matrix on `threads` host threads: the
    tensor amax first (one pass), then row ranges in parallel, each with that
    amax supplied, so every range gets the whole matrix's tensor scale.  The
    oracle's C code releases the interpreter lock while it runs."""
    if threads <= 1:
        orc.quantize(bits)
        return
    amax = float(np.abs(workloads.bf16_to_f32(bits)).max())
    bounds = np.linspace(0, bits.shape[0], threads + 1).astype(int)
    parts = [bits[a:b] for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
    list(pool.map(lambda part: orc.quantize(part, amax=amax), parts))


def cpu_oracle_rate(mats: dict, rows_per_matrix: int, threads: int = 1) -> tuple[float, str, float]:
    """Time the oracle on the first `rows_per_matrix` rows of each matrix, on
    `threads` host threads (row ranges)."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle

    oracle.build()
    subs = [np.ascontiguousarray(bits[:rows_per_matrix]) for bits in mats.values()]
    n = sum(s.size for s in subs)
    with ThreadPoolExecutor(max_workers=max(1, threads)) as pool:
        t0 = time.perf_counter()
        for sub in subs:
            oracle_quantize_threads(oracle, sub, threads, pool)
        dt = time.perf_counter() - t0
    sample = (f"first {rows_per_matrix} rows of each of the 7 matrices ({n / 1e6:.1f}M values), "
              f"{threads} thread{'s' if threads > 1 else ''}")
    return n / dt / 1e9, sample, dt


# ---------------------------------------------------------------- fos arm


def _events(torch, n):
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def _to_dev(torch, bits, dev):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)


def run_fos(args, dist: Dist) -> None:
    import torch

    import adaptive_quantization_fos_b300 as fos

    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    dist.init("nccl")
    stream = torch.cuda.current_stream()
    pk = peaks()

    mats_np = workloads.qwen3_8b_weights()
    # one batch per step, smallest matrix first (each launch takes the next
    # matrix's amax beside the current matrix's quantization)
    order = sorted(mats_np, key=lambda k: mats_np[k].size)
    mats = {k: _to_dev(torch, mats_np[k], dev) for k in order}
    bq = fos.BatchQuantizer([mats[k].shape for k in order], device=dev)
    xs = [mats[k] for k in order]
    elems = sum(v.numel() for v in mats.values())
    launches_per_step = 1  # the first matrix's amax pass
    for k in order:
        r, c = mats[k].shape
        # one quantize launch per matrix (chained), plus the pad fill of the
        # scale layout when the shape leaves padding
        launches_per_step += 1 + (1 if (r % 128 or (c // 16) % 4) else 0)

    def step():
        bq(xs)

    e0, e1 = _events(torch, 2)
    # the clock sampler starts before the warm-up: its thread's start-up then
    # does not compete with the timed region's first launches
    with ClockSampler(dev.index) as clk:
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        dist.barrier()
        torch.cuda.synchronize()
        h0 = time.perf_counter()
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        h1 = time.perf_counter()
        clk.mark(h0, h1)
        # the same steps, untimed, so that the clock record covers at least
        # 0.3 s of this load even when the timed region is a few ms
        while time.perf_counter() - h0 < 0.3:
            for _ in range(20):
                step()
            torch.cuda.synchronize()
    dist.barrier()
    t_ms = dist.max(e0.elapsed_time(e1), dev)
    ms_per_step = t_ms / args.steps
    value = dist.world * elems * args.steps / (t_ms * 1e-3) / 1e9

    # the step's kernels (the batch: the first matrix's amax pass and one
    # chained quantize launch per matrix, back to back on the launching
    # stream), timed by this rank's own CUDA events around the timed region:
    # the average quantize launch is a step's time over its 7 quantize
    # launches (the small amax launch of the first matrix overlaps the first)
    tot_t = e0.elapsed_time(e1)
    n_launch = args.steps * len(mats)
    achieved = elems * args.steps * BYTES_PER_ELEM_QUANT / (tot_t * 1e-3) / 1e9
    tpe = recorded_traffic_per_elem()
    roofline = {"bound": "hbm",
                "kernel": "quant_rows_kernel<4/6, RNE, 1D, chained> batch: per step 1 amax launch + 7 quantize "
                          "launches, each taking the next matrix's amax beside its quantization",
                "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / pk["hbm_gbs"], 4),
                "peak_source": pk["source"] + " copy bandwidth (hbm_gbs), burst",
                "bytes_per_elem": BYTES_PER_ELEM_QUANT,
                "traffic": None if tpe is None else round(tpe * elems / len(mats)),
                "traffic_note": "DRAM read+write bytes per quantize launch (a step's total over its 7 quantize "
                                "launches), from the committed warm-cache ncu capture of one batch call (all 8 "
                                "launches, amax re-reads included), scaled by values" if tpe else "no current capture",
                "algorithmic_bytes_per_launch": round(BYTES_PER_ELEM_QUANT * elems / len(mats)),
                "avg_launch_us": round(tot_t / n_launch * 1e3, 2),
                "timed": "CUDA events on the launching stream around the timed region; a step's time split "
                         "over its 7 quantize launches"}

    # context: the quantize pass alone (amax supplied), per-launch timing
    reps = max(3, min(args.steps, 100))
    amax = {k: fos.tensor_amax(v) for k, v in mats.items()}
    qk = {k: fos.Quantizer(*v.shape, device=dev, tensor_amax=amax[k]) for k, v in mats.items()}
    for k in mats:
        qk[k](mats[k])
    torch.cuda.synchronize()
    ev = _events(torch, 2 * reps * len(mats))
    i = 0
    for _ in range(reps):
        for k in mats:
            ev[i].record(stream)
            qk[k](mats[k])
            ev[i + 1].record(stream)
            i += 2
    torch.cuda.synchronize()
    tq = sum(ev[j].elapsed_time(ev[j + 1]) for j in range(0, len(ev), 2))
    roofline["quantize_pass_only"] = {
        "note": "amax supplied (opt->tensor_amax): the quantize pass alone, input read from HBM",
        "achieved": round(elems * reps * BYTES_PER_ELEM_QUANT / (tq * 1e-3) / 1e9, 1),
        "frac": round(elems * reps * BYTES_PER_ELEM_QUANT / (tq * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
        "avg_launch_us": round(tq / (reps * len(mats)) * 1e3, 2)}

    out = {"metric": METRIC, "value": round(value, 2), "unit": "Gelem/s", "n_gpus": dist.world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
           "data": "synthetic",
           "config": {"workload": WORKLOAD, "elements_per_step": elems, "input_bytes_per_step": 2 * elems,
                      "l2": "inputs larger than L2 (386 MB per step, 126 MB L2)",
                      "parallelism": f"replicas x{dist.world}" if dist.world > 1 else "single GPU",
                      "step_algorithmic_gbs": round(elems * BYTES_PER_ELEM_QUANT / (ms_per_step * 1e-3) / 1e9, 1)},
           "roofline": roofline, "gpu_launches": launches_per_step * args.steps, "clocks": clk.summary()}

    if not args.no_extras and dist.rank == 0:
        out["e2e"] = e2e_host_buffers(torch, fos, mats_np, dev, max(2, min(args.steps, 10)))
        out["secondary"] = secondary(torch, fos, dev, pk)
    if dist.rank == 0 and dist.world == 1 and not args.no_extras:
        cpu = host_cpu()
        rate1, sample1, secs1 = cpu_oracle_rate(mats_np, CPU_SAMPLE_ROWS, 1)
        rows_all = min(4096, CPU_SAMPLE_ROWS * max(1, cpu["nproc"] // 4))
        rate_n, sample_n, secs_n = cpu_oracle_rate(mats_np, rows_all, cpu["nproc"])
        out["cpu_baseline"] = {"value": round(rate_n, 6), "unit": "Gelem/s", "cores": cpu["nproc"], "kind": "oracle",
                               "sample": sample_n, "seconds": round(secs_n, 2), "cpu_model": cpu["model"],
                               "nproc": cpu["nproc"],
                               "single_thread": {"value": round(rate1, 6), "cores": 1, "sample": sample1,
                                                 "seconds": round(secs1, 2)}}
    if dist.rank == 0:
        print(json.dumps(out), flush=True)
    dist.close()


def e2e_host_buffers(torch, fos, mats_np, dev, steps) -> dict:
    """Same metric through the public API with host buffers: per step, copy
    each matrix host->device from pinned memory, quantize it, and copy its
    codes, scales and tensor scale back to pinned host memory.  Three streams
    pipeline the matrices: matrix i+1's upload overlaps matrix i's
    quantization and matrix i-1's download (PCIe is full duplex), and the next
    step's uploads start while this step's last matrices are still being
    quantized and downloaded.  Events order each buffer's reuse: a matrix is
    uploaded again only once the previous step's quantization has read it, and
    quantized again only once the previous step's download has read its
    outputs."""
    # largest first: the last matrix, whose download ends the step, is then the smallest
    order = sorted(mats_np, key=lambda k: -mats_np[k].size)
    host_in = {k: torch.from_numpy(mats_np[k].view(np.int16)).view(torch.bfloat16).pin_memory() for k in order}
    dev_in = {k: torch.empty(v.shape, dtype=torch.bfloat16, device=dev) for k, v in host_in.items()}
    qs = {k: fos.Quantizer(*v.shape, device=dev) for k, v in host_in.items()}
    host_out = {}
    for k, q in qs.items():
        o = q.out
        host_out[k] = (torch.empty(o.codes.shape, dtype=torch.uint8).pin_memory(),
                       torch.empty(o.sf.shape, dtype=torch.uint8).pin_memory(),
                       torch.empty(1, dtype=torch.float32).pin_memory())
    h2d = sum(v.numel() * 2 for v in host_in.values())
    d2h = sum(a.numel() + b.numel() + 4 for a, b, _ in host_out.values())
    s_in, s_q, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    main = torch.cuda.current_stream(dev)
    prev = {"q": {}, "out": {}}  # the previous step's events per matrix

    def step():
        ev_in, ev_q, ev_out = {}, {}, {}
        for k in order:
            if k in prev["q"]:
                s_in.wait_event(prev["q"][k])
            with torch.cuda.stream(s_in):
                dev_in[k].copy_(host_in[k], non_blocking=True)
                ev_in[k] = torch.cuda.Event()
                ev_in[k].record(s_in)
        for k in order:
            s_q.wait_event(ev_in[k])
            if k in prev["out"]:
                s_q.wait_event(prev["out"][k])
            qs[k](dev_in[k], stream=s_q)
            ev_q[k] = torch.cuda.Event()
            ev_q[k].record(s_q)
        for k in order:
            s_out.wait_event(ev_q[k])
            with torch.cuda.stream(s_out):
                o = qs[k].out
                a, b, c = host_out[k]
                a.copy_(o.codes, non_blocking=True)
                b.copy_(o.sf, non_blocking=True)
                c.copy_(o.tensor_scale, non_blocking=True)
                ev_out[k] = torch.cuda.Event()
                ev_out[k].record(s_out)
        prev["q"], prev["out"] = ev_q, ev_out

    def join():
        main.wait_stream(s_in)
        main.wait_stream(s_q)
        main.wait_stream(s_out)

    s_in.wait_stream(main)
    step()
    join()
    torch.cuda.synchronize()
    e0, e1 = _events(torch, 2)
    e0.record(main)
    for s in (s_in, s_q, s_out):
        s.wait_stream(main)
    for _ in range(steps):
        step()
    join()
    e1.record(main)
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) * 1e-3
    elems = sum(v.numel() for v in host_in.values())
    return {"value": round(elems * steps / t / 1e9, 3), "unit": "Gelem/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps,
            "note": "pinned host buffers; upload, quantize and download of the 7 matrices pipelined on 3 streams, "
                    "consecutive steps overlapped (each buffer reused only after its previous reader is done)"}


def _time_calls(torch, fn, reps: int) -> float:
    """Average ms per call of fn over reps (after one warm-up call)."""
    fn()
    torch.cuda.synchronize()
    e0, e1 = _events(torch, 2)
    e0.record()
    for _ in range(reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def _time_flushed(torch, flush, fn, reps: int) -> float:
    """Average ms of fn() alone with a cold L2: before each call a write of
    `flush` (larger than L2), then a short spin (torch.cuda._sleep, no memory
    traffic) that keeps the GPU busy while the host enqueues the start event
    and fn; CUDA events on the current stream bracket fn alone."""
    fn()
    torch.cuda.synchronize()
    ev = _events(torch, 2 * reps)
    for i in range(reps):
        flush.fill_(1)
        torch.cuda._sleep(100000)  # about 50 us at 2 GHz
        ev[2 * i].record()
        fn()
        ev[2 * i + 1].record()
    torch.cuda.synchronize()
    return sum(ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(reps)) / reps


def secondary(torch, fos, dev, pk) -> dict:
    res = {}
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # > L2, written before each call

    def measure(name, bits, reps=20, **opts):
        x = _to_dev(torch, bits, dev)
        q = fos.Quantizer(*x.shape, device=dev, **opts)

        t = _time_flushed(torch, flush, lambda: q(x), reps)
        n = x.numel()
        gbs = n * BYTES_PER_ELEM_QUANT / (t * 1e-3) / 1e9
        res[name] = {"ms": round(t, 4), "gelem_s": round(n / (t * 1e-3) / 1e9, 2),
                     "algorithmic_gbs": round(gbs, 1), "frac_of_hbm": round(gbs / pk["hbm_gbs"], 4),
                     "shape": list(x.shape), "options": {k: v for k, v in opts.items() if k != "tensor_amax"}}
        if delayed:
            # the same call with the tensor amax supplied (delayed scaling, a
            # previous step's amax): the quantize pass alone
            amax = fos.tensor_amax(x, hadamard=opts.get("hadamard", False), transpose=opts.get("transpose", False),
                                   hadamard_seed=opts.get("hadamard_seed", 0))
            qd = fos.Quantizer(*x.shape, device=dev, tensor_amax=amax, **opts)
            td = _time_flushed(torch, flush, lambda: qd(x), reps)
            gd = n * BYTES_PER_ELEM_QUANT / (td * 1e-3) / 1e9
            res[name]["amax_supplied"] = {"ms": round(td, 4), "gelem_s": round(n / (td * 1e-3) / 1e9, 2),
                                          "algorithmic_gbs": round(gd, 1), "frac_of_hbm": round(gd / pk["hbm_gbs"], 4)}

    delayed = True
    act = workloads.activations(16384, 4096, seed=3001)
    measure("activation_rht_rowmajor", act, hadamard=True, hadamard_seed=3002)
    measure("activation_rht_transposed", act, hadamard=True, hadamard_seed=3002, transpose=True)
    del act
    grad = workloads.gradients(8192, 12288, seed=4001)
    measure("gradient_sr_1d", grad, rounding=fos.FOS_ROUND_STOCHASTIC, sr_seed=4002)
    measure("gradient_sr_2d", grad, rounding=fos.FOS_ROUND_STOCHASTIC, sr_seed=4002, block_2d=True)
    measure("gradient_rne_2d", grad, block_2d=True)
    # MXFP4 with the 4/6 choice: no tensor scale, so one pass; 2 + 0.5 + 1/32
    # algorithmic bytes per value
    g = _to_dev(torch, grad, dev)
    mq = fos.quantize_mxfp4(g)  # outputs reused: the call below is the C entry point alone
    t = _time_flushed(torch, flush, lambda: fos.fos_quantize_mxfp4(
        g.data_ptr(), g.shape[0], g.shape[1], g.stride(0), fos.FOS_SCALE_4OVER6, mq.sf_layout, mq.codes.data_ptr(),
        mq.codes.stride(0), mq.scales.data_ptr(), 0, torch.cuda.current_stream().cuda_stream), 10)
    gbs = g.numel() * (2 + 0.5 + 1 / 32) / (t * 1e-3) / 1e9
    res["gradient_mxfp4"] = {"ms": round(t, 4), "gelem_s": round(g.numel() / (t * 1e-3) / 1e9, 2),
                             "algorithmic_gbs": round(gbs, 1), "frac_of_hbm": round(gbs / pk["hbm_gbs"], 4),
                             "shape": list(g.shape), "options": "MXFP4, 4/6 choice between the MX exponent and one "
                                                                "more, RNE, single pass"}
    del g, grad
    res["weights_layout_batch"] = weights_layout_batch(torch, fos, dev, pk, flush)
    res["linear_forward"] = linear_forward(torch, fos, dev, pk)
    res["linear_backward"] = linear_backward(torch, fos, dev, pk)
    return res


def weights_layout_batch(torch, fos, dev, pk, flush) -> dict:
    """The Qwen3-8B layer weight set quantized transposed (W^T, as the dgrad
    product reads it) and in 2D 16x16 tiles: one fos_quantize_batch call (one
    amax launch for all seven, then the seven quantize launches) against seven
    fos_quantize calls, each call or set timed with L2 flushed before it."""
    mats = workloads.qwen3_8b_weights()
    order = sorted(mats, key=lambda k: mats[k].size)
    xs = [_to_dev(torch, mats[k], dev) for k in order]
    n = sum(x.numel() for x in xs)
    out = {"values": n}
    for name, opts in (("transposed", dict(transpose=True)), ("2d", dict(block_2d=True))):
        bq = fos.BatchQuantizer([tuple(x.shape) for x in xs], device=dev, **opts)
        qs = [fos.Quantizer(*x.shape, device=dev, **opts) for x in xs]

        def separate():
            for q, x in zip(qs, xs):
                q(x)

        tb = _time_flushed(torch, flush, lambda: bq(xs), 10)
        ts = _time_flushed(torch, flush, separate, 10)
        gbs = n * BYTES_PER_ELEM_QUANT / (tb * 1e-3) / 1e9
        out[name] = {"batch_ms": round(tb, 4), "separate_calls_ms": round(ts, 4),
                     "gelem_s": round(n / (tb * 1e-3) / 1e9, 2), "algorithmic_gbs": round(gbs, 1),
                     "frac_of_hbm": round(gbs / pk["hbm_gbs"], 4), "options": opts}
        del bq, qs
    return out


def linear_backward(torch, fos, dev, pk) -> dict:
    """dX = dY W and dW = dY^T X for the linear forward's layer (X 8192 x 4096
    activations, W 12288 x 4096 weights) with dY 8192 x 12288 from the
    gradient recipe, through fos_linear_backward with the training recipe
    (SR on dY, RHT along M on the weight-gradient operands): four
    quantizations and two NVFP4 GEMMs per call."""
    M, N, K = 8192, 12288, 4096
    dy = _to_dev(torch, workloads.gradients(M, N, seed=6001), dev)
    x = _to_dev(torch, workloads.activations(M, K, seed=6002), dev)
    w = _to_dev(torch, workloads.student_t(N, K, seed=6003), dev)
    bw = fos.LinearBackward(M, N, K, device=dev, sr_seed=11, hadamard_seed=12)
    dx = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    dw = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
    try:
        bw(dy, x, w, dx=dx, dw=dw)
    except fos.FosError as e:
        return {"status": f"backward unavailable: {e}"}
    # the operands' quantization alone, to split the time
    qs = [fos.Quantizer(M, N, device=dev, rounding=fos.FOS_ROUND_STOCHASTIC, sr_seed=11),
          fos.Quantizer(N, K, device=dev, transpose=True),
          fos.Quantizer(M, N, device=dev, rounding=fos.FOS_ROUND_STOCHASTIC, sr_seed=11, transpose=True,
                        hadamard=True, hadamard_seed=12),
          fos.Quantizer(M, K, device=dev, transpose=True, hadamard=True, hadamard_seed=12)]
    srcs = [dy, w, dy, x]
    # the layer's two products on the operands it left in its workspace
    ops = bw.operands()
    with ClockSampler(dev.index) as clk:
        t = _time_calls(torch, lambda: bw(dy, x, w, dx=dx, dw=dw), 20)
        tg = _time_calls(torch, lambda: (fos.gemm(ops[0], ops[1], out=dx), fos.gemm(ops[2], ops[3], out=dw)), 20)
        tq = _time_calls(torch, lambda: [q(s) for q, s in zip(qs, srcs)], 20)
        names = ["dY_rows_sr", "Wt_cols", "dYt_cols_sr_rht", "Xt_cols_rht"]
        each = {n: round(_time_calls(torch, lambda q=q, s=s: q(s), 20), 4) for n, q, s in zip(names, qs, srcs)}
    flops = 2 * 2.0 * M * N * K
    return {"ms": round(t, 4), "gemm_ms": round(tg, 4), "quantize_ms": round(t - tg, 4),
            "quantize_note": "the layer's time less its two products: four quantizations, dY's two tensor "
                             "maxima taken from one read and its two stochastic-rounding quantizations from "
                             "one launch",
            "quantize_separate_calls_ms": round(tq, 4), "quantize_ms_each": each,
            "tflops_effective": round(flops / (t * 1e-3) / 1e12, 1),
            "gemm_tflops": round(flops / (tg * 1e-3) / 1e12, 1), "clocks": clk.summary(),
            "shape": {"M": M, "N": N, "K": K},
            "options": "SR on dY (both copies), RHT along M on dY^T and X^T, W^T 1D"}


def mma_rate(torch, fos, dev) -> dict:
    """The tensor-pipe throughput of the GEMM's own MMA instruction
    (kind::mxf4nvf4, E4M3 scales per 16 values, M = 128, K = 64, N = 128 or
    256) on this GPU: fos_selftest_mma_rate, one CTA per SM issuing MMAs back
    to back on operands resident in shared memory, timed with CUDA events."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    s = torch.cuda.current_stream(dev)
    out = {"sms": sms}
    iters = 1 << 15
    with ClockSampler(dev.index) as clk:
        for n in (256, 128):
            for it in (64, iters):  # a short warm-up launch, then the timed one
                e0, e1 = _events(torch, 2)
                e0.record(s)
                st = fos.fos_selftest_mma_rate(n, it, sms, status.data_ptr(), s.cuda_stream)
                e1.record(s)
                if st != fos.FOS_OK:
                    return {"status": f"probe unavailable (status {st})"}
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            out[f"n{n}"] = {"ms": round(ms, 3), "tflops": round(2.0 * 128 * n * 64 * 4 * iters * sms / (ms * 1e-3) / 1e12, 1)}
    out["timeout"] = int(status.item()) != 0
    out["clocks"] = clk.summary()
    out["instruction"] = "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X, M=128, K=64"
    return out


def linear_forward(torch, fos, dev, pk) -> dict:
    """Quantize A (8192 x 4096 activations) and W (12288 x 4096 weights) with
    4/6 1D RNE, then C = A W^T in NVFP4 on the tensor cores.  Also the whole
    layer through fos_linear_forward (A quantized, then the GEMM) against W
    quantized once beforehand."""
    A = _to_dev(torch, workloads.activations(8192, 4096, seed=5001), dev)
    W = _to_dev(torch, workloads.student_t(12288, 4096, seed=5002), dev)
    qa, qw = fos.Quantizer(*A.shape, device=dev), fos.Quantizer(*W.shape, device=dev)
    a, w = qa(A), qw(W)
    C = torch.empty((8192, 12288), dtype=torch.bfloat16, device=dev)
    try:
        fos.gemm(a, w, out=C)
    except fos.FosError as e:
        return {"status": f"gemm unavailable: {e}"}
    flops = 2.0 * 8192 * 12288 * 4096
    layer = fos.LinearForward(8192, 4096, device=dev)
    with ClockSampler(dev.index) as clk:
        t = _time_calls(torch, lambda: fos.gemm(a, w, out=C), 50)
        # the whole layer: X quantized (one-launch quantizer), then the GEMM as
        # its programmatic dependent; and the same two steps as separate calls
        t_layer = _time_calls(torch, lambda: layer(A, w, out=C), 50)
        t_two = _time_calls(torch, lambda: (qa(A), fos.gemm(a, w, out=C)), 50)
    tf = flops / (t * 1e-3) / 1e12
    fp4_peak = pk["bf16_tflops"] * 6.0  # measured bf16 burst x nominal dense fp4/bf16 ratio (13.5 / 2.25)
    rate = mma_rate(torch, fos, dev)
    # the same contraction from MXFP4 operands (E8M0 scales per 32 values)
    am, wm = fos.quantize_mxfp4(A), fos.quantize_mxfp4(W)
    try:
        fos.gemm_mxfp4(am, wm, out=C)
        with ClockSampler(dev.index) as clk_mx:
            t_mx = _time_calls(torch, lambda: fos.gemm_mxfp4(am, wm, out=C), 50)
        tf_mx = flops / (t_mx * 1e-3) / 1e12
        mx = {"gemm_ms": round(t_mx, 4), "tflops": round(tf_mx, 1), "clocks": clk_mx.summary(),
              "frac_of_mma_rate": round(tf_mx / rate["n256"]["tflops"], 4) if rate.get("n256") else None}
    except fos.FosError as e:
        mx = {"status": f"gemm_mxfp4 unavailable: {e}"}
    return {"gemm_ms": round(t, 4), "tflops": round(tf, 1), "clocks": clk.summary(),
            "mma_rate_probe": rate,
            "frac_of_mma_rate": round(tf / rate["n256"]["tflops"], 4) if rate.get("n256") else None,
            "gemm_mxfp4": mx,
            "layer_forward_ms": round(t_layer, 4), "layer_forward_tflops": round(flops / (t_layer * 1e-3) / 1e12, 1),
            "quantize_then_gemm_ms": round(t_two, 4),
            "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": round(fp4_peak, 1), "unit": "TFLOP/s",
                         "frac": round(tf / fp4_peak, 4),
                         "peak_source": "measured bf16 burst x 6 (nominal dense fp4/bf16 ratio)"}}


# ---------------------------------------------------------- reference arm


def run_reference(args, dist: Dist) -> None:
    if dist.rank != 0:
        return
    import oracle

    oracle.build()
    from concurrent.futures import ThreadPoolExecutor

    mats_np = workloads.qwen3_8b_weights()
    cpu = host_cpu()
    threads = cpu["nproc"]
    rows = REF_SAMPLE_ROWS * max(1, min(threads, 64) // 4)
    subs = {k: np.ascontiguousarray(v[:rows]) for k, v in mats_np.items()}
    n = sum(v.size for v in subs.values())
    pool = ThreadPoolExecutor(max_workers=threads)

    def step():
        for v in subs.values():
            oracle_quantize_threads(oracle, v, threads, pool)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    pool.shutdown()
    value = n * args.steps / dt / 1e9
    sample = (f"first {rows} rows of each of the 7 matrices per step ({n / 1e6:.2f}M values), {threads} threads "
              f"over row ranges ({cpu['model']})")
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "Gelem/s", "n_gpus": dist.world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
           "config": {"workload": WORKLOAD, "elements_per_step": n, "l2": "host run (no GPU)"},
           "cpu_baseline": {"value": round(value, 6), "unit": "Gelem/s", "cores": threads, "kind": "oracle",
                            "sample": sample, "cpu_model": cpu["model"], "nproc": cpu["nproc"]},
           "e2e": {"value": round(value, 6), "unit": "Gelem/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


# ------------------------------------------------------------ profiling


def run_case(args) -> None:
    """One small case for ncu: a few launches of one kernel, nothing else timed."""
    import torch

    import adaptive_quantization_fos_b300 as fos

    dev = torch.device("cuda", 0)
    if args.case == "quant_rows_chained":
        # the Qwen3-8B layer weight set as one batch (smallest first): the
        # chained quantize launches
        mats = workloads.qwen3_8b_weights()
        order = sorted(mats, key=lambda k: mats[k].size)
        xs = [_to_dev(torch, mats[k], dev) for k in order]
        bq = fos.BatchQuantizer([x.shape for x in xs], device=dev)
        for _ in range(2):
            bq(xs)
    elif args.case == "quant_cols_batch":
        # the same weight set quantized transposed as one batch call: one amax
        # launch for all seven, then one transposed quantize launch per matrix
        mats = workloads.qwen3_8b_weights()
        order = sorted(mats, key=lambda k: mats[k].size)
        xs = [_to_dev(torch, mats[k], dev) for k in order]
        bq = fos.BatchQuantizer([x.shape for x in xs], device=dev, transpose=True)
        for _ in range(2):
            bq(xs)
    elif args.case == "quant_rows_one_launch":
        # 12288 x 4096 bf16 (100.7 MB, the gate/up projection shape), no amax
        # supplied: the one-launch quantizer (amax pass, barrier, quantize pass)
        x = _to_dev(torch, workloads.student_t(12288, 4096, seed=9002), dev)
        q = fos.Quantizer(*x.shape, device=dev, one_launch=True)
        for _ in range(3):
            q(x)
    elif args.case == "quant_rows_two_launch":
        # the same matrix through the default form: amax pass, then the
        # quantize pass as its programmatic dependent
        x = _to_dev(torch, workloads.student_t(12288, 4096, seed=9002), dev)
        q = fos.Quantizer(*x.shape, device=dev)
        for _ in range(3):
            q(x)
    elif args.case == "quant_rows":
        # 12288 x 8192 bf16 (201 MB > L2), amax supplied: only the quantize kernel runs
        x = _to_dev(torch, workloads.student_t(12288, 8192, seed=9001), dev)
        amax = fos.tensor_amax(x)
        q = fos.Quantizer(*x.shape, device=dev, tensor_amax=amax)
        for _ in range(3):
            q(x)
    elif args.case == "quant_rows_sr":
        # 8192 x 12288 gradient (201 MB > L2), stochastic rounding, amax
        # supplied: only the row quantize kernel runs
        x = _to_dev(torch, workloads.gradients(8192, 12288, seed=4001), dev)
        amax = fos.tensor_amax(x)
        q = fos.Quantizer(*x.shape, device=dev, tensor_amax=amax, rounding=fos.FOS_ROUND_STOCHASTIC, sr_seed=4002)
        for _ in range(3):
            q(x)
    elif args.case == "quant_cols_sr_rht":
        # the same gradient transposed (blocks along its rows) with SR and the
        # RHT, amax supplied: only the transposed quantize kernel runs
        x = _to_dev(torch, workloads.gradients(8192, 12288, seed=4001), dev)
        amax = fos.tensor_amax(x, hadamard=True, transpose=True, hadamard_seed=12)
        q = fos.Quantizer(*x.shape, device=dev, tensor_amax=amax, rounding=fos.FOS_ROUND_STOCHASTIC, sr_seed=11,
                          transpose=True, hadamard=True, hadamard_seed=12)
        for _ in range(3):
            q(x)
    elif args.case == "quant_cols_rht":
        # the 16384 x 4096 activation transposed with the RHT, RNE, amax
        # supplied: only the transposed quantize kernel runs
        x = _to_dev(torch, workloads.activations(16384, 4096, seed=3001), dev)
        amax = fos.tensor_amax(x, hadamard=True, transpose=True, hadamard_seed=3002)
        q = fos.Quantizer(*x.shape, device=dev, tensor_amax=amax, hadamard=True, hadamard_seed=3002, transpose=True)
        for _ in range(3):
            q(x)
    elif args.case == "quant_rows_rht":
        # 16384 x 4096 activations with the RHT, amax supplied: only the row
        # quantize kernel runs
        x = _to_dev(torch, workloads.activations(16384, 4096, seed=3001), dev)
        amax = fos.tensor_amax(x, hadamard=True, hadamard_seed=3002)
        q = fos.Quantizer(*x.shape, device=dev, tensor_amax=amax, hadamard=True, hadamard_seed=3002)
        for _ in range(3):
            q(x)
    elif args.case == "quant_2d":
        # the 8192 x 12288 gradient in 16 x 16 tiles, RNE, amax supplied: only
        # the 2D quantize kernel runs
        x = _to_dev(torch, workloads.gradients(8192, 12288, seed=4001), dev)
        amax = fos.tensor_amax(x)
        q = fos.Quantizer(*x.shape, device=dev, tensor_amax=amax, block_2d=True)
        for _ in range(3):
            q(x)
    elif args.case == "quant_mxfp4":
        # 8192 x 12288 gradient (201 MB > L2), MXFP4 with the 4/6 choice: one
        # single-pass kernel
        x = _to_dev(torch, workloads.gradients(8192, 12288, seed=4001), dev)
        for _ in range(3):
            fos.quantize_mxfp4(x)
    elif args.case == "mma_rate":
        # the tensor-pipe rate probe: one CTA per SM issuing the GEMM's MMA
        # instruction back to back (N = 256), three launches
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        for _ in range(3):
            st = fos.fos_selftest_mma_rate(256, 4096, sms, 0, torch.cuda.current_stream().cuda_stream)
            if st != fos.FOS_OK:
                raise SystemExit(f"probe status {st}")
    elif args.case == "gemm":
        A = _to_dev(torch, workloads.activations(8192, 4096, seed=5001), dev)
        W = _to_dev(torch, workloads.student_t(12288, 4096, seed=5002), dev)
        a = fos.quantize(A)
        w = fos.quantize(W)
        C = torch.empty((8192, 12288), dtype=torch.bfloat16, device=dev)
        for _ in range(3):
            fos.gemm(a, w, out=C)
    elif args.case == "gemm_mx":
        # the same contraction from MXFP4 operands
        A = _to_dev(torch, workloads.activations(8192, 4096, seed=5001), dev)
        W = _to_dev(torch, workloads.student_t(12288, 4096, seed=5002), dev)
        a = fos.quantize_mxfp4(A)
        w = fos.quantize_mxfp4(W)
        C = torch.empty((8192, 12288), dtype=torch.bfloat16, device=dev)
        for _ in range(3):
            fos.gemm_mxfp4(a, w, out=C)
    elif args.case == "linear_backward":
        # the layer's backward at 8192 x 12288 x 4096 (SR on dY, RHT along M):
        # the fused dY quantization, W^T and X^T, the two GEMMs
        dy = _to_dev(torch, workloads.gradients(8192, 12288, seed=6001), dev)
        x = _to_dev(torch, workloads.activations(8192, 4096, seed=6002), dev)
        w = _to_dev(torch, workloads.student_t(12288, 4096, seed=6003), dev)
        bw = fos.LinearBackward(8192, 12288, 4096, device=dev, sr_seed=11, hadamard_seed=12)
        for _ in range(3):
            bw(dy, x, w)
    else:
        raise SystemExit(f"unknown case {args.case}")
    torch.cuda.synchronize()
    print(f"case {args.case} done")


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["fos", "reference"], default="fos")
    ap.add_argument("--no-extras", action="store_true", help="headline only (no e2e, secondary, CPU baseline)")
    ap.add_argument("--case", default=None, help="run one small profiling case instead of the benchmark")
    args = ap.parse_args()
    if args.case:
        run_case(args)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    dist = Dist()
    if args.gpus != dist.world and dist.world > 1:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE {dist.world}")
    if args.impl == "reference":
        run_reference(args, dist)
    else:
        run_fos(args, dist)


if __name__ == "__main__":
    main()
