"""Benchmark of the composite multi-LoRA delta on GB300.

One step = one pass of the whole hot path over one batch: build the mapping
from the batch's per-token pair lists (its CSR copy; the adapter-ordered
tuples too where the path reads them), then apply the fused delta
y += sum alpha (x A[:, :k]) B[:k, :] through the C ABI.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

Prints one JSON line.  `value` is tokens/s over the timed steps with every
input resident in HBM; the steps run from a captured CUDA graph and rotate
over R independent replicas (pool, x, y, pair lists, mapping) whose total size
exceeds twice the L2, so every step reads cold data from HBM.  `e2e` times the
same step through lora_delta_apply_host from pinned host buffers, with the
host->device copies of the step's inputs and the device->host copy of y
inside the timed region.  `roofline` measures lora_delta_apply alone (same
rotation) against the measured HBM copy bandwidth.  `--impl reference` times
the fp64 CPU oracle on the host cores instead (the reference arm).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "composite-LoRA delta tokens/s and achieved HBM GB/s vs GB300 peak, per config"
CONFIG_NAMES = {
    "distinct": "distinct decode, q_proj 4096x4096, r=8, T=32, 3 unshared adapters/token, pool 96",
    "zipf": "Zipf(1.5) decode, gate_proj 4096->14336, r=8, T=64, 2-4 adapters/token, pool 128",
    "prefill": "sparse MoE-LoRA prefill, 4096x4096, r=16, 16 requests lognormal lengths, top-2 of 8, pool 64",
    "sweep1": "rank sweep k_i~U{1..64}, k/v_proj 4096->1024, r_max=64, pool 1000, T=1",
    "sweep8": "rank sweep k_i~U{1..64}, k/v_proj 4096->1024, r_max=64, pool 1000, T=8",
    "sweep64": "rank sweep k_i~U{1..64}, k/v_proj 4096->1024, r_max=64, pool 1000, T=64",
    "sweep256": "rank sweep k_i~U{1..64}, k/v_proj 4096->1024, r_max=64, pool 1000, T=256",
}
PATH_NAMES = {0: "auto", 1: "split", 2: "fused", 3: "mma", 4: "decode"}
# kernels of lora_delta_apply per path (the mapping's CSR stage adds one
# launch per step; the paths that read the adapter-sorted tuples launch the
# sort stage first, which returns at once when the build is sorted already)
PATH_KERNELS = {
    "split": (2, "sort stage + k_shrink + k_expand (PDL)"),
    "fused": (1, "k_dec_fused (cooperative, one launch)"),
    "mma": (2, "sort stage + k_mma_shrink + k_mma_expand (tcgen05, PDL)"),
    "decode": (2, "k_dec_shrink + k_dec_expand (PDL)"),
}
SORTED_PATHS = ("split", "mma")


def sort_stage_kernels(P: int, capacity: int) -> int:
    """Kernels of the mapping's sort stage: two (count, scatter) for batches
    of 2048..32768 pairs over pools of at most 1024 slots whose per-CTA
    counts fit in shared memory, else one (the one-CTA sort)."""
    ctas = (P + 511) // 512
    return 2 if P >= 2048 and ctas <= 64 and capacity <= 1024 and ctas * capacity * 4 <= 200 * 1024 else 1


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# kernel sources of each path's apply kernels (besides the shared headers)
PATH_SOURCES = {
    "decode": ["decode.cu"],
    "mma": ["mma.cu", "tcgen05.cuh"],
    "split": ["shrink.cu", "shrink_core.cuh", "expand.cu", "expand_core.cuh"],
    "fused": ["fused.cu", "shrink_core.cuh", "expand_core.cuh"],
}
SHARED_SOURCES = ["internal.h", "ptx.cuh"]


_C_TOKENS = re.compile(r'//[^\n]*|/\*.*?\*/|"(?:\\.|[^"\\])*"|\'(?:\\.|[^\'\\])*\'', re.S)


def code_only(text: str) -> str:
    """C/C++/CUDA source with comments removed and whitespace collapsed (string
    and character literals kept): what the compiler sees, so that an edit of
    the documentation does not count as a change of the kernels."""
    text = _C_TOKENS.sub(lambda mt: " " if mt.group(0).startswith("/") else mt.group(0), text)
    return " ".join(text.split())


def path_source_files(path: str) -> list:
    """Repository-relative files a path's apply kernels are built from."""
    files = sorted(set(PATH_SOURCES[path] + SHARED_SOURCES))
    return [f"tenant_composite_lora_gb300/csrc/{f}" for f in files] + ["include/lora.h"]


def sources_digest(path: str, read=None) -> str:
    """Digest of the code (comments aside) a path's apply kernels are built
    from, the ABI header included: a traffic figure taken with other code no
    longer describes the kernels.  `read(relpath) -> str` defaults to this
    checkout."""
    read = read or (lambda rel: open(os.path.join(ROOT, rel), encoding="utf-8").read())
    h = hashlib.sha256()
    for rel in path_source_files(path):
        h.update(rel.encode())
        h.update(code_only(read(rel)).encode())
    return h.hexdigest()[:16]


def ncu_traffic(config: str, path: str):
    """dram bytes (read + write) per lora_delta_apply, summed over the apply's
    kernels, from a committed ncu summary; valid only while the path's kernel
    sources are unchanged."""
    fp = os.path.join(ROOT, "profiles", f"traffic_{config}_{path}.txt")
    if not os.path.exists(fp):
        return None
    kv = {}
    for line in open(fp):
        if ":" in line:
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    if kv.get("sources_sha256_16") != sources_digest(path):
        return None
    try:
        return int(kv["dram_bytes_per_apply"])
    except (KeyError, ValueError):
        return None


class NvmlClocks:
    """SM clock and clock-event reasons read through NVML (the driver's
    libnvidia-ml), polled from a thread: fine-grained enough for timed
    regions of a few milliseconds.  Reading only; no setting is changed."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index: int):
        import ctypes
        import threading
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.dev = ctypes.c_void_p()
        found = False
        try:  # the CUDA device by UUID (NVML indexes ignore CUDA_VISIBLE_DEVICES)
            import torch
            uuid = str(torch.cuda.get_device_properties(cuda_index).uuid)
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            found = self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.dev)) == 0
        except Exception:
            found = False
        if not found:
            n = ctypes.c_uint()
            self.lib.nvmlDeviceGetCount_v2(ctypes.byref(n))
            idx = 0 if n.value == 1 else cuda_index
            if self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(idx), ctypes.byref(self.dev)) != 0:
                raise RuntimeError("no NVML handle")
        mx = ctypes.c_uint()
        self.lib.nvmlDeviceGetMaxClockInfo(self.dev, 1, ctypes.byref(mx))  # 1 = SM clock
        self.max_mhz = float(mx.value)
        self.reason_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.sm, self.bits = [], 0
        self.stop_flag = threading.Event()
        self.thread = threading.Thread(target=self._run, daemon=True)

    def sample(self):
        c = self.ct.c_uint()
        r = self.ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.dev, 1, self.ct.byref(c)) == 0:
            self.sm.append(float(c.value))
        if self.reason_fn(self.dev, self.ct.byref(r)) == 0:
            self.bits |= int(r.value)

    def _run(self):
        while not self.stop_flag.is_set():
            self.sample()
            time.sleep(0.0005)

    def start(self):
        self.sample()
        self.thread.start()

    def stop(self) -> dict:
        self.stop_flag.set()
        self.thread.join(timeout=5)
        self.sample()
        reasons = sorted(v for k, v in self.REASONS.items() if self.bits & k)
        return {"sm_mhz": statistics.median(self.sm) if self.sm else None, "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(self.sm), "source": "nvml"}


class ClockSampler:
    """Clock / throttle samples during the timed region: NVML when the driver
    library loads, else nvidia-smi."""

    def __init__(self, index: int):
        self.proc = None
        self.nvml = None
        try:
            self.nvml = NvmlClocks(index)
            self.nvml.start()
            return
        except Exception:
            self.nvml = None
        self.path = os.path.join(tempfile.gettempdir(), f"tclora_clocks_{os.getpid()}.csv")
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(index), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.nvml is not None:
            return self.nvml.stop()
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvidia-smi"}


def dist_setup(n):
    if n <= 1 or "RANK" not in os.environ:
        return 0, 1, None
    import torch.distributed as dist
    dist.init_process_group("nccl" if os.environ.get("TCL_BENCH_BACKEND") != "gloo" else "gloo")
    return dist.get_rank(), dist.get_world_size(), dist


def max_over_ranks(x, dist, device=None):
    """The maximum of a float over all ranks (the float itself on one rank)."""
    if dist is None:
        return x
    import torch
    dev = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def pass_times_ms(replay, passes: int, stream, event_cls) -> list:
    """Device time of each of `passes` consecutive replays, from events
    recorded on the stream between them (one event per boundary)."""
    evs = [event_cls(enable_timing=True) for _ in range(passes + 1)]
    evs[0].record(stream)
    for i in range(passes):
        replay()
        evs[i + 1].record(stream)
    evs[-1].synchronize()
    return [evs[i].elapsed_time(evs[i + 1]) for i in range(passes)]


def spread(values_us: list) -> dict:
    """Median, p10 and p90 of per-step times (microseconds)."""
    v = np.asarray(values_us, np.float64)
    return {"p10": round(float(np.percentile(v, 10)), 3), "median": round(float(np.median(v)), 3),
            "p90": round(float(np.percentile(v, 90)), 3), "samples": int(v.size)}


def bench_ours(args, rank, world, dist):
    import torch
    import tenant_composite_lora_gb300 as tcl
    from tenant_composite_lora_gb300 import native
    import workloads as W
    from workloads.device import bf16_tensor, bf16_to_numpy_bits

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    wl = W.make(args.config)
    ab = W.algorithmic_bytes(wl)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    R = max(2, int(np.ceil(2.0 * l2 / max(ab["total"], 1))))
    R = min(R, args.max_replicas)

    with torch.cuda.stream(stream):
        # replicas: pools registered from the same factors, separate buffers
        A_t = [bf16_tensor(wl.A[a], dev) for a in range(wl.capacity)]
        B_t = [bf16_tensor(wl.B[a], dev) for a in range(wl.capacity)]
        reps = []
        for r in range(R):
            pool = tcl.LoraPool(wl.d_in, wl.d_out, wl.r_max, wl.capacity)
            for a in range(wl.capacity):
                pool.register(a, A_t[a], B_t[a], int(wl.ranks[a]))
            mp = tcl.LoraMapping(wl.T, wl.P, wl.capacity)
            rep = dict(pool=pool, mapping=mp,
                       off=torch.from_numpy(wl.offsets).to(dev), ids=torch.from_numpy(wl.ids).to(dev),
                       alpha=torch.from_numpy(wl.alpha).to(dev), x=bf16_tensor(wl.x, dev),
                       y0=bf16_tensor(wl.y, dev), y=bf16_tensor(wl.y, dev))
            reps.append(rep)
        del A_t, B_t
        torch.cuda.synchronize()

        def step(rep):
            native.lora_build_mapping(rep["mapping"].handle, rep["off"], rep["ids"], rep["alpha"],
                                      wl.T, wl.P, stream)
            native.lora_delta_apply_path(rep["x"], rep["y"], rep["pool"].handle, None, rep["mapping"].handle,
                                         args.path_id, stream)

        def apply_only(rep):
            native.lora_delta_apply_path(rep["x"], rep["y"], rep["pool"].handle, None, rep["mapping"].handle,
                                         args.path_id, stream)

        # correctness spot check of replica 0 (one step from y0)
        reps[0]["y"].copy_(reps[0]["y0"])
        step(reps[0])
        stream.synchronize()
        st = native.lora_mapping_status(reps[0]["mapping"].handle, stream)
        if st != 0:
            raise RuntimeError(f"device status {st}")

        # graphs: one pass over all replicas, and the first K mod R replicas
        # for the remainder, so that exactly K steps are timed
        def capture(fn, n=None):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for rep in reps[: (R if n is None else n)]:
                    fn(rep)
            return g

        for rep in reps:  # build every mapping once before the apply-only graph
            native.lora_build_mapping(rep["mapping"].handle, rep["off"], rep["ids"], rep["alpha"],
                                      wl.T, wl.P, stream)
        K = max(1, args.steps)
        full, rem = divmod(K, R)
        g_step = capture(step)
        g_apply = capture(apply_only)
        g_step_rem = capture(step, rem) if rem else None
        g_apply_rem = capture(apply_only, rem) if rem else None
        stream.synchronize()

        def timed(graph, graph_rem):
            """Device time of exactly K steps: `full` replays of the pass and
            one of the remainder, after W warm-up passes, with a barrier and a
            synchronisation on both sides; the maximum over ranks."""
            for _ in range(max(1, args.warmup)):
                graph.replay()
            stream.synchronize()
            if dist is not None:
                dist.barrier()
            torch.cuda.synchronize(dev)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(full):
                graph.replay()
            if graph_rem is not None:
                graph_rem.replay()
            e1.record(stream)
            e1.synchronize()
            torch.cuda.synchronize(dev)
            return max_over_ranks(e0.elapsed_time(e1), dist, dev)

        clk = ClockSampler(local)
        ms_step_total = timed(g_step, g_step_rem)
        clocks = clk.stop()
        steps_done = K
        ms_per_step = ms_step_total / steps_done
        ms_apply = timed(g_apply, g_apply_rem) / steps_done
        passes = max(1, full)

        # spread of the step time: each pass (R steps, one per replica) timed on
        # its own, after the contract's timed region; reported per step
        try:
            n_pass = min(max(passes, 20), 200)
            spread_step = spread([ms * 1e3 / R for ms in pass_times_ms(g_step.replay, n_pass, stream,
                                                                        torch.cuda.Event)])
            spread_step["steps_per_sample"] = R
        except Exception as exc:  # an auxiliary figure never costs the line itself
            spread_step = {"error": f"{type(exc).__name__}: {exc}"}

        # end to end through the host entry point (pinned buffers, copies timed)
        x_h = torch.from_numpy(wl.x.view(np.int16).copy()).pin_memory()
        y_h = torch.from_numpy(wl.y.view(np.int16).copy()).pin_memory()
        off_h = torch.from_numpy(wl.offsets).pin_memory()
        ids_h = torch.from_numpy(wl.ids).pin_memory()
        al_h = torch.from_numpy(wl.alpha).pin_memory()
        rep = reps[0]
        for _ in range(max(1, args.warmup)):
            native.lora_delta_apply_host(x_h, y_h, off_h, ids_h, al_h, wl.T, wl.P, rep["pool"].handle, None,
                                         rep["mapping"].handle, stream)
        stream.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)
        e2e_steps = max(args.steps, 10)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h0 = time.perf_counter()
        for _ in range(e2e_steps):
            native.lora_delta_apply_host(x_h, y_h, off_h, ids_h, al_h, wl.T, wl.P, rep["pool"].handle, None,
                                         rep["mapping"].handle, stream)
        host_us = (time.perf_counter() - h0) * 1e6 / e2e_steps  # the calls' own host time (enqueue)
        e1.record(stream)
        e1.synchronize()
        ms_e2e = max_over_ranks(e0.elapsed_time(e1), dist, dev) / e2e_steps
        h2d = wl.x.nbytes + wl.y.nbytes + wl.offsets.nbytes + wl.ids.nbytes + wl.alpha.nbytes
        d2h = wl.y.nbytes

    peak, peak_kind = peaks()
    path_taken = args.path if args.path_id != 0 else PATH_NAMES[
        native.lora_dispatch_choose(wl.T, wl.P, wl.r_max, wl.d_in, wl.d_out)]
    n_apply_kernels, kernel_desc = PATH_KERNELS[path_taken]
    if path_taken in SORTED_PATHS:
        n_apply_kernels += sort_stage_kernels(wl.P, wl.capacity)
    achieved = ab["total"] / (ms_apply * 1e-3) / 1e9
    value = world * wl.T / (ms_per_step * 1e-3)
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": steps_done,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded numpy draws shaped like the pages' workloads)",
        "config": {
            "workload": args.config, "desc": CONFIG_NAMES.get(args.config, args.config),
            "T": wl.T, "P": wl.P, "d_in": wl.d_in, "d_out": wl.d_out, "r_max": wl.r_max,
            "pool": wl.capacity, "distinct_adapters": ab["U"], "sum_k": ab["sum_k"],
            "step": "lora_build_mapping + lora_delta_apply",
            "path": path_taken if args.path_id != 0 else f"auto -> {path_taken}",
            "l2_protocol": f"inputs larger than L2: {R} rotating replicas, {R * ab['total'] / 1e6:.0f} MB "
                           f"touched per pass vs {l2 / 1e6:.0f} MB L2",
            "parallelism": "replicas only" if world > 1 else "single GPU",
        },
        "roofline": {
            "bound": "hbm", "kernel": f"lora_delta_apply = {kernel_desc}",
            "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
            "algorithmic_bytes": ab["total"], "apply_us": round(ms_apply * 1e3, 3),
            "traffic": ncu_traffic(args.config, path_taken),
        },
        "e2e": {"value": round(world * wl.T / (ms_e2e * 1e-3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms_e2e, 6),
                "api": "lora_delta_apply_host", "host_us_per_call": round(host_us, 3)},
        "gpu_launches": (1 + n_apply_kernels) * steps_done,  # the CSR stage is one launch
        "clocks": clocks,
        "step_us_spread": spread_step,
    }
    return line, wl


class ColdTimer:
    """Device time of a captured piece of work with a cold L2: every timed
    replay runs a graph [read of FLUSH_BYTES, work]; a graph of the read
    alone is timed the same way and subtracted, so the figure is the work's
    own time starting from an L2 that holds none of its data."""

    FLUSH_BYTES = 256 << 20  # twice the L2

    def __init__(self, torch, stream, device):
        self.torch, self.stream, self.dev = torch, stream, device
        self.src = torch.empty(self.FLUSH_BYTES // 4, dtype=torch.float32, device=device).fill_(1.0)
        self.out = torch.empty((), dtype=torch.float32, device=device)
        self.g_flush = self.capture(lambda: None)
        self.flush_ms = None

    def capture(self, fn):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            torch.sum(self.src, dim=0, out=self.out)
            fn()
        return g

    def _mean_ms(self, g, n):
        torch = self.torch
        for _ in range(3):
            g.replay()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        for _ in range(n):
            g.replay()
        e1.record(self.stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / n

    def time_us(self, fn, n=100):
        g = self.capture(fn)
        with self.torch.cuda.stream(self.stream):
            a = self._mean_ms(g, n)
            b = self._mean_ms(self.g_flush, n)
            a2 = self._mean_ms(g, n)
            b2 = self._mean_ms(self.g_flush, n)
        return max(0.0, ((a + a2) - (b + b2)) / 2 * 1e3)

    def time_spread_us(self, fn, n=100, blocks=10):
        """As time_us (2n replays of the work, 2n of the read alone), in
        `blocks` alternating blocks: the mean and the spread of the blocks."""
        g = self.capture(fn)
        per = max(1, (2 * n) // blocks)
        with self.torch.cuda.stream(self.stream):
            return cold_blocks_us(lambda: self._mean_ms(g, per), lambda: self._mean_ms(self.g_flush, per), blocks)


def cold_blocks_us(work_ms, flush_ms, blocks: int):
    """Alternate `blocks` times a block of [read, work] replays (work_ms():
    its mean ms per replay) with a block of the read alone (flush_ms()); the
    work's own time per block is the difference.  Returns the mean over the
    blocks (microseconds, at least 0) and their median, p10 and p90."""
    diffs = []
    for _ in range(blocks):
        a = work_ms()
        b = flush_ms()
        diffs.append((a - b) * 1e3)
    return max(0.0, float(np.mean(diffs))), spread(diffs)


def per_config_lines(args, peak, torch, stream, dev):
    """Every workload of the metric: the apply and the step (mapping +
    apply) from a cold L2, tokens/s, achieved HBM bandwidth against the
    measured peak, and the ncu traffic of the path when it is on file."""
    from tenant_composite_lora_gb300 import native
    import workloads as W
    from workloads.device import DeviceWorkload
    timer = ColdTimer(torch, stream, dev)
    out = {}
    for name in ["distinct", "zipf", "prefill", "sweep1", "sweep8", "sweep64", "sweep256"]:
        t0 = time.perf_counter()
        wl = W.make(name)
        ab = W.algorithmic_bytes(wl)
        with torch.cuda.stream(stream):
            dw = DeviceWorkload(wl, stream=stream)
            try:
                y = dw.y0.clone()
                m, pool = dw.mapping.handle, dw.pool.handle

                def apply_():
                    native.lora_delta_apply(dw.x, y, pool, None, m, stream)

                def step_():
                    native.lora_build_mapping(m, dw.offsets, dw.ids, dw.alpha, wl.T, wl.P, stream)
                    native.lora_delta_apply(dw.x, y, pool, None, m, stream)

                apply_us, apply_sp = timer.time_spread_us(apply_)
                step_us, step_sp = timer.time_spread_us(step_)
            finally:
                dw.close()
        path = PATH_NAMES[native.lora_dispatch_choose(wl.T, wl.P, wl.r_max, wl.d_in, wl.d_out)]
        achieved = ab["total"] / (apply_us * 1e-6) / 1e9 if apply_us > 0 else None
        out[name] = {
            "T": wl.T, "P": wl.P, "path": path, "apply_us": round(apply_us, 3), "step_us": round(step_us, 3),
            "tokens_per_s": round(wl.T / (step_us * 1e-6), 1) if step_us > 0 else None,
            "algorithmic_bytes": ab["total"], "achieved_gbs": round(achieved, 1) if achieved else None,
            "frac": round(achieved / peak, 4) if achieved else None, "traffic": ncu_traffic(name, path),
            "apply_us_blocks": apply_sp, "step_us_blocks": step_sp,
            "setup_s": round(time.perf_counter() - t0, 2),
        }
    return {"protocol": "cold L2: a 256 MB read before every timed replay, its own time subtracted; "
                        "mean over 200 replays in 10 blocks of 20, alternating with blocks of the read "
                        "alone (*_blocks: median, p10, p90 of the blocks); path = the dispatch table's",
            "configs": out}


def ablation_lines(torch, stream, dev):
    """The pages' kernel ablation on this GPU: the fused path against the
    naive per-adapter loop, Copy + SGMV and the explicit pre-merge, each
    timed eagerly from a cold L2 (events around the call; the naive loop and
    Copy + SGMV read the batch's segments back to the host inside the call)."""
    import tenant_composite_lora_gb300 as tcl
    from tenant_composite_lora_gb300 import native
    import workloads as W
    from workloads.device import DeviceWorkload
    flush = torch.empty(ColdTimer.FLUSH_BYTES // 4, dtype=torch.float32, device=dev).fill_(1.0)
    out = {}
    for name in ["distinct", "zipf"]:
        wl = W.make(name)
        res = {}
        with torch.cuda.stream(stream):
            dw = DeviceWorkload(wl, stream=stream)
            try:
                y = dw.y0.clone()
                nb = max(native.lora_ablation_workspace_bytes(v, wl.T, wl.P, wl.d_in, wl.d_out, wl.r_max)
                         for v in (1, 2, 3))
                ws = torch.empty(nb, dtype=torch.uint8, device=dev)
                calls = {
                    "fused_path": lambda: native.lora_delta_apply(dw.x, y, dw.pool.handle, None, dw.mapping.handle,
                                                                  stream),
                    "naive_loop": lambda: native.lora_delta_apply_ablation(dw.x, y, dw.pool.handle, None,
                                                                           dw.mapping.handle, 1, ws, nb, stream),
                    "copy_sgmv": lambda: native.lora_delta_apply_ablation(dw.x, y, dw.pool.handle, None,
                                                                          dw.mapping.handle, 2, ws, nb, stream),
                    "premerge": lambda: native.lora_delta_apply_ablation(dw.x, y, dw.pool.handle, None,
                                                                         dw.mapping.handle, 3, ws, nb, stream),
                }
                for key, fn in calls.items():
                    times = []
                    for it in range(8):
                        torch.sum(flush)
                        stream.synchronize()
                        e0 = torch.cuda.Event(enable_timing=True)
                        e1 = torch.cuda.Event(enable_timing=True)
                        e0.record(stream)
                        fn()
                        e1.record(stream)
                        e1.synchronize()
                        if it >= 2:
                            times.append(e0.elapsed_time(e1) * 1e3)
                    res[key] = round(statistics.median(times), 2)
                del ws
            finally:
                dw.close()
        base = res["fused_path"]
        res["ratio_to_fused"] = {k: round(v / base, 2) for k, v in res.items() if k != "fused_path"}
        out[name] = res
    return {"unit": "us per apply (eager, cold L2, median of 6)", "workloads": out,
            "pages_claim": "fused ~1/2 of Copy+SGMV and ~1/5 of the naive loop (DyMerge-LoRA, L40, Fig 16)"}


def multi_projection_lines(torch, stream, dev):
    """One layer's q, k, v, o projections (Llama-3-8B shapes, r = 8) over the
    distinct decode batch: lora_delta_apply_multi against four separate
    lora_delta_apply calls, cold L2."""
    import tenant_composite_lora_gb300 as tcl
    from tenant_composite_lora_gb300 import native
    import workloads as W
    from workloads.device import bf16_tensor
    base = W.make("distinct")
    timer = ColdTimer(torch, stream, dev)
    shapes = {"q": (4096, 4096), "k": (4096, 1024), "v": (4096, 1024), "o": (4096, 4096)}
    rng = np.random.default_rng(5)
    pools, xs, ys = [], [], []
    m = tcl.LoraMapping(base.T, base.P, base.capacity)
    try:
        with torch.cuda.stream(stream):
            for _, (d_in, d_out) in shapes.items():
                p = tcl.LoraPool(d_in, d_out, 8, base.capacity)
                for a in range(base.capacity):
                    A = torch.randn(d_in, 8, device=dev).mul_(0.02).to(torch.bfloat16)
                    B = torch.randn(8, d_out, device=dev).mul_(0.02).to(torch.bfloat16)
                    p.register(a, A, B, 8, stream)
                pools.append(p)
                xs.append(bf16_tensor(W.f32_to_bf16_bits(rng.standard_normal((base.T, d_in)).astype(np.float32) * 0.02),
                                      dev))
                ys.append(torch.zeros(base.T, d_out, dtype=torch.bfloat16, device=dev))
            m.build(torch.from_numpy(base.offsets).to(dev), torch.from_numpy(base.ids).to(dev),
                    torch.from_numpy(base.alpha).to(dev), stream)
            stream.synchronize()
            projs = [(x, y, p.handle, None) for x, y, p in zip(xs, ys, pools)]
            multi = timer.time_us(lambda: native.lora_delta_apply_multi(projs, m.handle, stream))
            separate = timer.time_us(lambda: [native.lora_delta_apply(x, y, p, None, m.handle, stream)
                                              for x, y, p, _ in projs])
    finally:
        for p in pools:
            p.close()
        m.close()
    return {"projections": {k: f"{v[0]}->{v[1]}, r=8" for k, v in shapes.items()}, "batch": "distinct decode",
            "multi_us": round(multi, 3), "separate_us": round(separate, 3),
            "per_projection_us": {"multi": round(multi / 4, 3), "separate": round(separate / 4, 3)}}


def recompress_lines(torch, stream, dev):
    """Recompression of one Llama-3-8B-shaped adapter (32 layers x q, k, v,
    o, gate, up, down at r = 16: 224 LoRA matrices) by lora_recompress, one
    call per projection shape, then the spectral rank policy; seconds and
    matrices per second, with the pages' whole-fleet figure as context."""
    import tenant_composite_lora_gb300 as tcl
    from tenant_composite_lora_gb300 import native
    shapes = {"q": (4096, 4096), "k": (4096, 1024), "v": (4096, 1024), "o": (4096, 4096),
              "gate": (4096, 14336), "up": (4096, 14336), "down": (14336, 4096)}
    L, r = 32, 16
    g = torch.Generator(device=dev).manual_seed(0)
    bufs = []
    with torch.cuda.stream(stream):
        for name, (d_in, d_out) in shapes.items():
            A = (torch.randn(L, d_in, r, device=dev, generator=g) * 0.02).to(torch.bfloat16)
            B = (torch.randn(L, r, d_out, device=dev, generator=g) * 0.02).to(torch.bfloat16)
            F = torch.empty(L, d_in, r, dtype=torch.float32, device=dev)
            T = torch.empty(L, r, d_out, dtype=torch.float32, device=dev)
            sig = torch.empty(L, r, dtype=torch.float32, device=dev)
            nb = native.lora_recompress_workspace_bytes(L, d_in, r)
            ws = torch.empty(nb, dtype=torch.uint8, device=dev)
            bufs.append((name, d_in, d_out, A, B, F, T, sig, ws, nb))

        def run():
            for name, d_in, d_out, A, B, F, T, sig, ws, nb in bufs:
                native.lora_recompress(A, B, L, d_in, d_out, r, F, T, sig, ws, nb, stream)

        run()
        stream.synchronize()
        times = []
        for _ in range(5):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            run()
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1))
        t0 = time.perf_counter()
        sig_all = np.concatenate([b[7].cpu().numpy() for b in bufs])
        cost = np.concatenate([np.full(L, b[1] + b[2], np.int32) for b in bufs])
        k = native.lora_rank_allocate(sig_all, np.full(sig_all.shape[0], r, np.int32), cost,
                                      native.LORA_RANK_SPECTRAL, 4, 1)
        alloc_ms = (time.perf_counter() - t0) * 1e3
    ms = statistics.median(times)
    n = L * len(shapes)
    return {"matrices": n, "r": r, "device_ms": round(ms, 3), "matrices_per_s": round(n / (ms * 1e-3), 1),
            "rank_allocation_host_ms": round(alloc_ms, 3), "mean_retained_rank": round(float(k.mean()), 3),
            "context": "pages: whole Llama35 fleet (7,840 matrices) in 2.06 s with FlashTSQR on one GH200 "
                       "(LoRAForge page, Sec. 6.3); random synthetic factors here"}


# Dispatch sweep: batches of T tokens with two pairs each, grouped into
# requests of `share` consecutive tokens that use the same two adapters of
# their own (share = 1: every token its own adapters, as in a decode batch;
# larger: prompt-like runs), or two distinct Zipf(1.5) draws over 128
# adapters per token ("zipf"); q_proj shape, every rank r_max.
SWEEP_T = [16, 64, 128, 256, 384, 512, 1024, 2048, 4096, 8192]
SWEEP_R = [8, 16, 32, 64]
SWEEP_SHARE = ["1", "16", "256", "zipf"]
SWEEP_PATHS = {"decode": 4, "split": 1, "mma": 3}
SWEEP_CAPACITY = 4096


def sweep_ids(T: int, share: str, rng) -> np.ndarray:
    """Adapter ids [T, 2] of the sweep's batch."""
    if share == "zipf":
        w = 1.0 / np.arange(1, 129) ** 1.5
        w /= w.sum()
        return np.stack([rng.choice(128, size=2, replace=False, p=w) for _ in range(T)]).astype(np.int32)
    s = int(share)
    req = np.arange(T) // s
    return (np.stack([2 * req, 2 * req + 1], axis=1) % SWEEP_CAPACITY).astype(np.int32)


def dispatch_sweep(torch, stream, dev) -> dict:
    """apply (and build + apply) time of every path on every sweep point,
    cold L2, with the dispatch table's own pick beside the fastest."""
    import tenant_composite_lora_gb300 as tcl
    from tenant_composite_lora_gb300 import native
    timer = ColdTimer(torch, stream, dev)
    d_in = d_out = 4096
    rng = np.random.default_rng(11)
    g = torch.Generator(device=dev).manual_seed(3)
    tmax = max(SWEEP_T)
    points = []
    with torch.cuda.stream(stream):
        x = (torch.randn(tmax, d_in, device=dev, generator=g) * 0.02).to(torch.bfloat16)
        y = torch.zeros(tmax, d_out, dtype=torch.bfloat16, device=dev)
        for r in SWEEP_R:
            pool = tcl.LoraPool(d_in, d_out, r, SWEEP_CAPACITY)
            A = (torch.randn(d_in, r, device=dev, generator=g) * 0.02).to(torch.bfloat16)
            B = (torch.randn(r, d_out, device=dev, generator=g) * 0.02).to(torch.bfloat16)
            for a in range(SWEEP_CAPACITY):
                pool.register(a, A, B, r, stream)
            try:
                for T in SWEEP_T:
                    for share in SWEEP_SHARE:
                        ids = sweep_ids(T, share, rng)
                        P = 2 * T
                        off = torch.arange(0, P + 1, 2, dtype=torch.int32, device=dev)
                        ids_d = torch.from_numpy(ids.reshape(-1)).to(dev)
                        al_d = torch.full((P,), 0.5, dtype=torch.float32, device=dev)
                        m = tcl.LoraMapping(T, P, SWEEP_CAPACITY)
                        xs, ys = x[:T], y[:T]
                        pt = {"T": T, "r": r, "share": share, "P": P, "U": int(np.unique(ids).size)}
                        try:
                            m.build(off, ids_d, al_d, stream)
                            for name, pid in SWEEP_PATHS.items():
                                def apply_(pid=pid):
                                    native.lora_delta_apply_path(xs, ys, pool.handle, None, m.handle, pid, stream)

                                def step_(pid=pid):
                                    native.lora_build_mapping(m.handle, off, ids_d, al_d, T, P, stream)
                                    native.lora_delta_apply_path(xs, ys, pool.handle, None, m.handle, pid, stream)
                                try:
                                    apply_()
                                    stream.synchronize()
                                except Exception as exc:  # a path that does not take this shape
                                    pt[name] = None
                                    pt[name + "_error"] = type(exc).__name__
                                    continue
                                n = 100 if T <= 512 else 30
                                pt[name] = round(timer.time_us(apply_, n), 2)
                                pt[name + "_step"] = round(timer.time_us(step_, n), 2)
                        finally:
                            m.close()
                        timed = {k: pt[k] for k in SWEEP_PATHS if pt.get(k) is not None}
                        pt["fastest"] = min(timed, key=timed.get)
                        pt["chosen"] = PATH_NAMES[native.lora_dispatch_choose(T, P, r, d_in, d_out)]
                        points.append(pt)
            finally:
                pool.close()
        del x, y
        # the metric's workloads on every path
        import workloads as W
        from workloads.device import DeviceWorkload
        configs = {}
        for name in ["distinct", "zipf", "prefill", "sweep1", "sweep8", "sweep64", "sweep256"]:
            wl = W.make(name)
            dw = DeviceWorkload(wl, stream=stream)
            res = {"T": wl.T, "P": wl.P, "r": wl.r_max,
                   "chosen": PATH_NAMES[native.lora_dispatch_choose(wl.T, wl.P, wl.r_max, wl.d_in, wl.d_out)]}
            try:
                yb = dw.y0.clone()
                for pname, pid in SWEEP_PATHS.items():
                    def apply_(pid=pid):
                        native.lora_delta_apply_path(dw.x, yb, dw.pool.handle, None, dw.mapping.handle, pid, stream)
                    apply_()
                    stream.synchronize()
                    res[pname] = round(timer.time_us(apply_, 100 if wl.T <= 512 else 30), 2)
            finally:
                dw.close()
            res["fastest"] = min(SWEEP_PATHS, key=lambda k: res[k])
            configs[name] = res
    return {"shape": f"{d_in}x{d_out}", "pairs_per_token": 2, "capacity": SWEEP_CAPACITY,
            "protocol": "cold L2 (256 MB read before every replay, its time subtracted); us per call",
            "points": points, "configs": configs}


def sweep_markdown(d: dict) -> str:
    """The sweep as the committed table (profiles/dispatch_sweep.md)."""
    paths = list(SWEEP_PATHS)
    out = ["# Dispatch sweep: every path's apply time over tokens x rank x adapter sharing", "",
           "Command (one GB300, after `python -c \"import __graft_entry__ as g; g.build()\"`):",
           "`python bench.py --dispatch-sweep --markdown > profiles/dispatch_sweep.md`", "",
           f"Shape {d['shape']} (Llama-3-8B q_proj), {d['pairs_per_token']} pairs per token (alpha 0.5), "
           f"pool of {d['capacity']} slots, every adapter at k = r.  share = tokens of a request: runs of that "
           "many consecutive tokens use the same two adapters of their own (1: every token its own, as in "
           "decode; larger: prompt-like); zipf = two distinct Zipf(1.5) draws over 128 adapters per token.  "
           f"Times: {d['protocol']}.  U = distinct adapters.", "",
           "| T | r | share | P | U | " + " | ".join(f"{p} us" for p in paths) + " | fastest | chosen | chosen / fastest |",
           "|" + "---|" * (8 + len(paths))]
    for p in d["points"]:
        t = {k: p.get(k) for k in paths}
        best = p["fastest"]
        ratio = (t[p["chosen"]] / t[best]) if t.get(p["chosen"]) and t[best] else None
        out.append(f"| {p['T']} | {p['r']} | {p['share']} | {p['P']} | {p['U']} | "
                   + " | ".join("-" if t[k] is None else f"{t[k]:.2f}" for k in paths)
                   + f" | {best} | {p['chosen']} | " + ("-" if ratio is None else f"{ratio:.2f}") + " |")
    out += ["", "## The metric's workloads, every path", "",
            "| workload | T | P | r | " + " | ".join(f"{p} us" for p in paths) + " | fastest | chosen |",
            "|" + "---|" * (6 + len(paths))]
    for name, c in d["configs"].items():
        out.append(f"| {name} | {c['T']} | {c['P']} | {c['r']} | " + " | ".join(f"{c[k]:.2f}" for k in paths)
                   + f" | {c['fastest']} | {c['chosen']} |")
    return "\n".join(out) + "\n"


def cpu_model() -> str:
    """The host CPU's name as the OS reports it ("unknown" when it does not)."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":", 1)[0].strip().lower()
                if key in ("model name", "cpu model", "hardware") and ":" in line:
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine() or "unknown"


def oracle_baseline(wl, budget_s: float):
    """The oracle as it stands on the host cores: whole batches with OpenMP
    over tokens for most of the budget, then a bounded single-thread sample
    (evenly spaced tokens) for the single-core figure."""
    import oracle
    th = oracle.max_threads()
    t0 = time.perf_counter()
    n = 0
    tokens = 0
    # whole batches while the budget lasts (at least one)
    while True:
        oracle.apply_workload(wl, threads=th, want_acc=False)
        n += 1
        tokens += wl.T
        if time.perf_counter() - t0 >= 0.8 * budget_s:
            break
    dt = time.perf_counter() - t0
    # single thread: a token sample sized from the measured rate (an estimate),
    # repeated until about a fifth of the budget has passed
    per_token_1 = dt * th / max(tokens, 1)
    n1 = int(min(wl.T, max(1, 0.2 * budget_s / max(per_token_1, 1e-9))))
    toks = np.linspace(0, wl.T - 1, n1).round().astype(np.int64)
    reps = 0
    t1 = time.perf_counter()
    while True:
        oracle.apply_tokens(wl, toks, threads=1)
        reps += 1
        if time.perf_counter() - t1 >= 0.2 * budget_s:
            break
    dt1 = time.perf_counter() - t1
    return {"value": round(tokens / dt, 3), "unit": "tokens/s", "cores": th, "kind": "oracle",
            "sample": f"{n} full batch(es) of the workload ({tokens} tokens, fp64, OpenMP over tokens)",
            "seconds": round(dt, 2), "cpu_model": cpu_model(), "nproc": os.cpu_count(),
            "single_thread": {"value": round(reps * n1 / dt1, 3), "unit": "tokens/s",
                              "sample": f"{reps} x {n1} evenly spaced tokens of the batch, fp64, one thread",
                              "seconds": round(dt1, 2)}}


def bench_reference(args):
    """The reference arm: the fp64 oracle on the host cores, W untimed and K
    timed steps, each step a bounded sample of the workload's tokens (the
    whole batch when it fits) sized so that the run takes about --ref-seconds (90 s by default)."""
    import oracle
    import workloads as W
    wl = W.make(args.config)
    th = oracle.max_threads()
    budget = max(0.002, args.ref_seconds / (args.steps + args.warmup))  # seconds per step
    n0 = min(wl.T, 16)
    t0 = time.perf_counter()
    oracle.apply_tokens(wl, np.arange(n0), threads=th)
    per_token = (time.perf_counter() - t0) / n0
    n = int(min(wl.T, max(1, budget / max(per_token, 1e-9))))
    if n >= wl.T:
        n = wl.T
        step = lambda: oracle.apply_workload(wl, threads=th, want_acc=False)
        sample = f"whole batch ({wl.T} tokens) per step"
    else:
        toks = np.linspace(0, wl.T - 1, n).round().astype(np.int64)
        step = lambda: oracle.apply_tokens(wl, toks, threads=th)
        sample = f"{n} of the batch's {wl.T} tokens (evenly spaced) per step"
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = args.steps * n / dt
    cb = {"value": round(value, 3), "unit": "tokens/s", "cores": th, "kind": "oracle",
          "sample": sample + ", fp64, OpenMP over tokens", "seconds": round(dt, 2),
          "cpu_model": cpu_model(), "nproc": os.cpu_count()}
    return {"metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.config, "desc": CONFIG_NAMES[args.config]}, "impl": "reference",
            "cpu_baseline": cb,
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="distinct", choices=sorted(CONFIG_NAMES))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=90.0,
                    help="wall time the reference arm aims for over its warm-up and timed steps")
    ap.add_argument("--max-replicas", type=int, default=64)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the per-config, ablation and multi-projection figures")
    ap.add_argument("--path", default="auto", choices=["auto", "split", "fused", "mma", "decode"],
                    help="force an execution path (default: the library's dispatch table)")
    ap.add_argument("--dispatch-sweep", action="store_true",
                    help="time every path over tokens x rank x adapter sharing and print that table instead")
    ap.add_argument("--markdown", action="store_true", help="with --dispatch-sweep: the table as Markdown")
    args = ap.parse_args()
    args.path_id = {"auto": 0, "split": 1, "fused": 2, "mma": 3, "decode": 4}[args.path]
    args.warmup = max(3, args.warmup)

    if args.impl == "reference":
        # the CPU oracle needs no process group: rank 0 alone runs and prints
        if int(os.environ.get("RANK", "0")) == 0:
            print(json.dumps(bench_reference(args)))
        return

    if args.dispatch_sweep:
        import torch
        dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
        torch.cuda.set_device(dev)
        d = dispatch_sweep(torch, torch.cuda.Stream(device=dev), dev)
        print(sweep_markdown(d) if args.markdown else json.dumps(d), end="" if args.markdown else "\n")
        return

    rank, world, dist = dist_setup(args.gpus)

    line, wl = bench_ours(args, rank, world, dist)
    if rank == 0:
        if not args.no_extras and world == 1:
            import torch
            dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
            stream = torch.cuda.Stream(device=dev)
            peak, _ = peaks()
            for key, fn in (("per_config", lambda: per_config_lines(args, peak, torch, stream, dev)),
                            ("ablation", lambda: ablation_lines(torch, stream, dev)),
                            ("multi_projection", lambda: multi_projection_lines(torch, stream, dev)),
                            ("recompress", lambda: recompress_lines(torch, stream, dev))):
                try:
                    line[key] = fn()
                except Exception as exc:  # an auxiliary figure never costs the line itself
                    line[key] = {"error": f"{type(exc).__name__}: {exc}"}
                torch.cuda.empty_cache()
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = oracle_baseline(wl, args.cpu_seconds)
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
