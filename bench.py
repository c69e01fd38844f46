#!/usr/bin/env python3
"""Benchmark of the frame-wise Gated DeltaNet forward on one B300 per rank.

Workload (one step = one full forward pass of a GDN layer): B=1, H=20, D=112,
F=121 latent frames x N=880 tokens (a 60 s 720p latent video: 961 raw frames at
8x temporal compression, a 40 x 22 latent grid per frame), bf16 q/k/v/o, fp32
beta/gamma/state, synthetic seeded inputs resident in HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line on rank 0.  ``value`` is tokens/s over all ranks (each rank
runs the whole workload on its own GPU: chains are independent, so ranks share
nothing on the data path -> weak scaling).  ``--impl reference`` times the fp64
CPU oracle on the host cores instead (the only other implementation of the
method), on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GDN fwd tokens/sec at 20 heads×D112; TFLOPS / HBM GB/s as % of B300 roofline"
WORKLOAD = "layer_60s_720p"
PEAKS_FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


# ----------------------------------------------------------------- arithmetic
def algorithmic(B, H, F, N, D):
    """Algorithmic bytes and flops of one forward (inputs read once, outputs written once)."""
    fh = B * H * F
    tok_bytes = N * D * 2
    stats_bytes = fh * (2 * tok_bytes + 4 * N)        # k, v, beta
    out_bytes = fh * (2 * tok_bytes + 4)              # q, o, gamma
    state_bytes = B * H * D * D * 4 * 2               # S_in, S_out
    flops = fh * (6 * N * D * D + 2 * D ** 3)
    return {"stats": stats_bytes, "out": out_bytes, "state": state_bytes,
            "total": stats_bytes + out_bytes + state_bytes, "flops": flops}


def step_bytes(B, H, N, D):
    """Algorithmic bytes of one streaming call: q, k, v, o, beta, gamma and the state in and out."""
    return B * H * (N * D * 2 * 4 + 4 * N + 4) + 2 * B * H * D * D * 4


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


def source_hash():
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(ROOT, "gated_deltanet_wise_b300", "csrc", "*"))):
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, if it matches this source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        d = json.load(fh)
    if d.get("source_hash") != source_hash():
        return None
    k = d.get("kernels", {}).get(kernel)
    return None if k is None else k.get("dram_bytes_per_launch_full")


# ------------------------------------------------------------- clock sampling
class ClockSampler:
    """Samples SM clocks and clock-event reasons (read-only) while the timed region runs.

    NVML (the driver's libnvidia-ml.so.1, through ctypes) is polled every ~2 ms
    on a thread; the device is found by PCI bus id, since NVML numbers every GPU
    of the machine.  If NVML cannot be loaded, ``nvidia-smi`` runs as a
    subprocess instead, and the sampler waits for its first sample before the
    timed region starts.  Nothing here changes a GPU setting.
    """

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
               0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}
    NVML_CLOCK_SM = 1

    def __init__(self, device):
        import torch
        self.samples, self.reasons, self.max_mhz, self.error = [], 0, None, None
        self._stop = threading.Event()
        self._th = None
        self._proc = None
        self.bus = None
        try:
            props = torch.cuda.get_device_properties(device)
            self.bus = "%08X:%02X:%02X.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
        except Exception as e:  # pragma: no cover - depends on the torch build
            self.error = f"pci id: {e}"
        self.nv = None
        try:
            import ctypes
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise RuntimeError("nvmlInit_v2 failed")
            h = ctypes.c_void_p()
            if self.bus is None or nv.nvmlDeviceGetHandleByPciBusId_v2(self.bus.encode(), ctypes.byref(h)) != 0:
                raise RuntimeError("no NVML handle for this device")
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self._reason_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self.nv, self.h, self._ct = nv, h, ctypes
        except Exception as e:
            self.error = f"nvml: {e}"

    def _run(self):
        ct, nv = self._ct, self.nv
        clk, rsn = ct.c_uint(), ct.c_ulonglong()
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(self.h, self.NVML_CLOCK_SM, ct.byref(clk)) == 0:
                self.samples.append(clk.value)
            if self._reason_fn(self.h, ct.byref(rsn)) == 0:
                self.reasons |= rsn.value
            time.sleep(0.002)

    def __enter__(self):
        if self.nv:
            self._th = threading.Thread(target=self._run, daemon=True)
            self._th.start()
            return self
        import subprocess
        import tempfile
        self._log = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        cmd = ["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits", "-lms", "20"]
        if self.bus:
            cmd += ["-i", self.bus]
        try:
            self._proc = subprocess.Popen(cmd, stdout=self._log, stderr=subprocess.DEVNULL)
            t0 = time.time()
            while time.time() - t0 < 5.0 and os.path.getsize(self._log.name) == 0:
                time.sleep(0.01)
        except Exception as e:
            self.error = f"nvidia-smi: {e}"
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self._th:
            self._th.join()
        if self._proc:
            self._proc.terminate()
            self._proc.wait()
            self._log.seek(0)
            bits = {"hw_slowdown": 0x8, "hw_thermal_slowdown": 0x40, "sw_thermal_slowdown": 0x20, "sw_power_cap": 0x4}
            for line in self._log.read().splitlines():
                f = [x.strip() for x in line.split(",")]
                if len(f) < 6:
                    continue
                try:
                    self.samples.append(float(f[0]))
                    self.max_mhz = float(f[1])
                except ValueError:
                    continue
                for n, v in zip(bits, f[2:6]):
                    if v.lower() == "active":
                        self.reasons |= bits[n]

    def summary(self):
        out = {"sm_mhz": statistics.median(self.samples) if self.samples else None, "sm_max_mhz": self.max_mhz,
               "reasons": [n for bit, n in self.REASONS.items() if self.reasons & bit and n != "gpu_idle"],
               "samples": len(self.samples), "source": "nvml" if self.nv else "nvidia-smi"}
        if not self.samples:
            out["error"] = self.error or "no samples"
        return out


# ---------------------------------------------------------------- CPU oracle
def oracle_sample(x, heads, frames):
    """Run the oracle on `heads` whole chains over the first `frames` frames; returns seconds."""
    import oracle
    N = x.N
    sl = slice(0, frames * N)
    args = (x.q[:, sl, :heads].contiguous(), x.k[:, sl, :heads].contiguous(), x.v[:, sl, :heads].contiguous(),
            x.beta[:, sl, :heads].contiguous(), x.gamma[:, :frames, :heads].contiguous(), None)
    args = [oracle._f32(a) if a is not None else None for a in args]
    t0 = time.perf_counter()
    oracle.frame_fwd(*args, N=N)
    return time.perf_counter() - t0


def cpu_baseline(x, target_s=15.0):
    """Oracle timed on the host cores on a bounded sample; value in full-layer tokens/s."""
    import oracle
    threads = oracle.num_threads()
    heads = x.H
    t1 = oracle_sample(x, heads, 1)
    frames = max(1, min(x.F, int(target_s / max(t1, 1e-3))))
    t = oracle_sample(x, heads, frames) if frames > 1 else t1
    tokens_equiv = frames * x.N * heads / x.H          # tokens of the 20-head layer
    return {"value": tokens_equiv / t, "unit": "tokens/s", "cores": min(threads, heads), "kind": "oracle",
            "sample": f"{heads} of {x.H} heads x first {frames} of {x.F} frames x {x.N} tokens, fp64, "
                      f"{t:.1f} s; scaled to 20-head tokens",
            "seconds": t}


# ----------------------------------------------------------------- our arm
def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, value):
    """The slowest rank's time (every rank gets it); NCCL groups reduce on the GPU, others on the CPU."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measure_streaming(x, K, W, stream):
    """121 single-frame gdn_frame_step calls carrying S (one pass of the streaming layer).

    Timed twice: replaying a CUDA graph that holds the F calls (the way a frame
    loop is meant to run) and as eager launches.  Returns the numbers for one
    pass and for one call.
    """
    import torch
    from gated_deltanet_wise_b300 import gdn
    B, H, F, N, D = x.B, x.H, x.F, x.N, x.D
    assert B == 1, "frame slices of the [B][F*N][H][D] tensors are contiguous only for B = 1"
    S = torch.empty(B, H, D, D, dtype=torch.float32, device=x.q.device)
    o = torch.empty_like(x.q)
    S0 = x.S0 if x.S0 is not None else torch.zeros_like(S)
    tok = N * H * D

    def ptr(t, off_elems):
        return t.data_ptr() + off_elems * t.element_size()

    L = gdn.lib()
    cs = torch.cuda.Stream(device=x.q.device)  # graphs are captured on a non-default stream
    sp = gdn._stream(cs)

    def one_pass():
        for f in range(F):
            s_in = S0.data_ptr() if f == 0 else S.data_ptr()   # the state is carried in place
            st = L.gdn_frame_step(ptr(x.q, f * tok), ptr(x.k, f * tok), ptr(x.v, f * tok),
                                  ptr(x.beta, f * N * H), ptr(x.gamma, f * H), s_in, S.data_ptr(),
                                  ptr(o, f * tok), B, H, N, D, 0.0, None, 0, sp)
            if st != gdn.GDN_OK:
                raise gdn.GdnError(st, "gdn_frame_step")

    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(cs):
        for _ in range(W):
            one_pass()
        torch.cuda.synchronize()
        t0.record(cs)
        for _ in range(K):
            one_pass()
        t1.record(cs)
        torch.cuda.synchronize()
        eager_ms = t0.elapsed_time(t1) / K
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cs):
            one_pass()
        for _ in range(W):
            g.replay()
        torch.cuda.synchronize()
        t0.record(cs)
        for _ in range(K):
            g.replay()
        t1.record(cs)
        torch.cuda.synchronize()
        graph_ms = t0.elapsed_time(t1) / K
    if gdn.gdn_device_status() != gdn.GDN_OK:
        raise RuntimeError("device status reports a timed-out wait")
    peaks, kind = load_peaks()
    call_bytes = step_bytes(B, H, N, D)
    call_us = graph_ms * 1e3 / F
    achieved = call_bytes / (call_us * 1e-6) / 1e9
    return {"workload": "streaming_60s_720p", "frames": F, "calls_per_pass": F, "kernel": "k4_frame_step_kernel",
            "graph_ms_per_pass": round(graph_ms, 4), "eager_ms_per_pass": round(eager_ms, 4),
            "us_per_call_graph": round(call_us, 3), "us_per_call_eager": round(eager_ms * 1e3 / F, 3),
            "tokens_per_s_graph": round(B * F * N / (graph_ms * 1e-3), 1),
            "algorithmic_bytes_per_call": call_bytes,
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": ncu_traffic("k4_frame_step_kernel"),
                         "kernel": "k4_frame_step_kernel",
                         "note": f"per call inside the graph (launch gaps included); peak {kind}"},
            "launches_per_pass": F}


def run_streaming_line(args):
    """Main line for the streaming workload: one step = one pass of F single-frame calls."""
    import torch
    from gated_deltanet_wise_b300.inputs import make_workload
    world, rank, local = dist_setup(args)
    dev = torch.device("cuda", torch.cuda.current_device())
    x = make_workload(args.workload, device=dev, seed=rank, F=args.frames)
    stream = torch.cuda.current_stream()
    barrier(world)
    with ClockSampler(dev) as clk:
        r = measure_streaming(x, args.steps, args.warmup, stream)
    barrier(world)
    ms = max_over_ranks(world, r["graph_ms_per_pass"])
    if rank == 0:
        line = {"metric": METRIC, "value": round(world * x.B * x.F * x.N / (ms * 1e-3), 1), "unit": "tokens/s",
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic",
                "config": {"workload": args.workload, "B": x.B, "H": x.H, "D": x.D, "F": x.F, "N": x.N,
                           "step": f"{x.F} gdn_frame_step calls carrying S, replayed as one CUDA graph",
                           "l2": "each call streams 17.9 MB of distinct frame data; the 1.9 GB pass exceeds L2"},
                "roofline": r["roofline"], "streaming": r, "gpu_launches": x.F * args.steps,
                "clocks": clk.summary()}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_ours(args):
    import torch
    from gated_deltanet_wise_b300 import gdn
    from gated_deltanet_wise_b300.inputs import make_workload

    world, rank, local = dist_setup(args)
    dev = torch.device("cuda", torch.cuda.current_device())
    x = make_workload(args.workload, device=dev, seed=rank, F=args.frames)
    B, H, F, N, D = x.B, x.H, x.F, x.N, x.D
    o = torch.empty_like(x.q)
    S_out = torch.empty(B, H, D, D, dtype=torch.float32, device=dev)
    nbytes = gdn.gdn_frame_fwd_workspace_size(B, H, F, N, D)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    K, W = args.steps, args.warmup

    def step(events=None):
        if events is None:  # the public entry point, as a user calls it
            st = gdn.gdn_frame_fwd(x.q, x.k, x.v, x.beta, x.gamma, x.S0, S_out, o, B, H, F, N, D, 0.0,
                                   ws, nbytes, stream)
        else:  # same launches with CUDA events between the three kernels
            st = gdn.gdn_frame_fwd_profiled(x.q, x.k, x.v, x.beta, x.gamma, x.S0, S_out, o, B, H, F, N, D, 0.0,
                                            ws, nbytes, events, stream)
        if st != gdn.GDN_OK:
            raise gdn.GdnError(st, "gdn_frame_fwd")

    for _ in range(W):
        step()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for e in (t0, t1):
        e.record(stream)  # creates the CUDA events outside the timed region
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(dev) as clk:
        t0.record(stream)
        for i in range(K):
            step()
        t1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    if gdn.gdn_device_status() != gdn.GDN_OK:
        raise RuntimeError("device status reports a timed-out wait")
    ms = t0.elapsed_time(t1) / K
    ms_max = max_over_ranks(world, ms)
    # per-kernel durations: a separate pass with events between the kernels (which
    # also keeps each kernel from overlapping its neighbour's tail)
    Kp = max(3, min(K, 50))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(Kp)]
    for row in ev:
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    for i in range(Kp):
        step(ev[i])
    torch.cuda.synchronize()
    stage_ms = [statistics.fmean(e[j].elapsed_time(e[j + 1]) for e in ev) for j in range(3)]

    alg = algorithmic(B, H, F, N, D)
    tokens = B * F * N
    value = world * tokens / (ms_max * 1e-3)
    peaks, peaks_kind = load_peaks()
    # dominant kernel: frame statistics (k, v, beta) or scan + output (q, o, gamma)
    names = ["k1_frame_stats_kernel", "k1b_chunk_boundary_kernel", "k2_scan_output_kernel"]
    kbytes = [alg["stats"], alg["state"], alg["out"]]
    dom = 0 if stage_ms[0] >= stage_ms[2] else 2
    achieved = kbytes[dom] / (stage_ms[dom] * 1e-3) / 1e9
    traffic = ncu_traffic(names[dom])
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic, "kernel": names[dom],
                "peak_source": f"{peaks_kind} STREAM-style copy (MEASURED_PEAKS.json hbm_gbs)",
                "algorithmic_bytes_per_launch": kbytes[dom],
                "stage_ms": {n: round(t, 5) for n, t in zip(names, stage_ms)},
                "stage_steps": Kp,
                "path": {"achieved_gbs": round(alg["total"] / (ms * 1e-3) / 1e9, 1),
                         "frac": round(alg["total"] / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                         "tflops": round(alg["flops"] / (ms * 1e-3) / 1e12, 2),
                         "tensor_frac": round(alg["flops"] / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4)}}

    variants = measure_variants(x, max(3, min(K, 30)), stream, alg, peaks)
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(x, K, W, world)
    streaming = None
    if not args.no_stream:
        from gated_deltanet_wise_b300.inputs import make_workload as mw
        xs = mw("streaming_60s_720p", device=dev, seed=rank)
        streaming = measure_streaming(xs, max(3, min(K, 20)), 3, stream)
        del xs
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(x)
    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": K,
                "warmup": W, "ms_per_step": round(ms_max, 5), "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": args.workload, "B": B, "H": H, "D": D, "F": F, "N": N, "tokens": tokens,
                           "l2": f"inputs {alg['total'] / 1e9:.2f} GB per step > 126 MB L2; no flush needed",
                           "parallelism": f"replica x{world} (independent chains per rank)"},
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": 3 * K,
                "streaming": streaming, "variants": variants,
                "clocks": clk.summary()}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def measure_variants(x, K, stream, alg, peaks):
    """The same layer through gdn_frame_fwd_ex: the token-ordered (product) reading,
    the reverse-direction scan and the fused chained scan (one cooperative launch
    after a memset of its hop flags), K back-to-back calls each after 3 warm-ups."""
    import torch
    from gated_deltanet_wise_b300 import gdn
    B, H, F, N, D = x.B, x.H, x.F, x.N, x.D
    o = torch.empty_like(x.q)
    S_out = torch.empty(B, H, D, D, dtype=torch.float32, device=x.q.device)
    out = {}
    for name, flags, launches in (("product", gdn.GDN_FWD_PRODUCT, 5), ("reverse", gdn.GDN_FWD_REVERSE, 3),
                                  ("fused", gdn.GDN_FWD_FUSED, 1)):
        nb = gdn.gdn_frame_fwd_ex_workspace_size(B, H, F, N, D, flags)
        ws = torch.empty(nb, dtype=torch.uint8, device=x.q.device)

        def step():
            st = gdn.gdn_frame_fwd_ex(x.q, x.k, x.v, x.beta, x.gamma, x.S0, S_out, o, B, H, F, N, D, 0.0, flags,
                                      ws, nb, stream)
            if st != gdn.GDN_OK:
                raise gdn.GdnError(st, "gdn_frame_fwd_ex")

        for _ in range(3):
            step()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0.record(stream)
        for _ in range(K):
            step()
        t1.record(stream)
        torch.cuda.synchronize()
        if gdn.gdn_device_status() != gdn.GDN_OK:
            raise RuntimeError("device status reports a timed-out wait")
        ms = t0.elapsed_time(t1) / K
        out[name] = {"ms_per_step": round(ms, 5), "tokens_per_s": round(B * F * N / (ms * 1e-3), 1),
                     "path_frac_hbm": round(alg["total"] / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                     "steps": K, "gpu_launches_per_step": launches}
        del ws
    out["backward"] = measure_backward(x, max(3, min(K, 10)), stream, peaks)
    out["block"] = measure_block(x, max(3, min(K, 10)), stream, peaks)
    out["context_parallel"] = measure_context_parallel(x, max(3, min(K, 20)), stream)
    return out


def measure_context_parallel(x, K, stream, world=2):
    """Frame-split context parallelism with the ranks' work run one after another on this GPU.
    Per rank: its composite pass over its frames (gdn_frame_composite; on the last rank, whose
    composites no rank composes, the statistics pass alone), its start state composed from the
    earlier ranks' composites onto S_in (gdn_state_compose once per earlier rank; the all-gather
    that carries the composites between GPUs is not in it) and the rest of its forward from the
    statistics in its workspace (gdn_frame_fwd_resume), against gdn_frame_fwd over the same
    frames from the same start state.  K calls each after 3 warm-ups; `ratio` is the largest
    rank's time over its plain forward."""
    import torch
    from gated_deltanet_wise_b300 import gdn
    from gated_deltanet_wise_b300.context_parallel import frame_split
    B, H, F, N, D = x.B, x.H, x.F, x.N, x.D
    dev = x.q.device

    def part(t, f0, f1, per_frame):
        return t[:, f0 * per_frame:f1 * per_frame].contiguous()

    def timed(fn):
        for _ in range(3):
            fn()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0.record(stream)
        for _ in range(K):
            fn()
        t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / K

    def ok(st, what):
        if st != gdn.GDN_OK:
            raise gdn.GdnError(st, what)

    gathered = []  # (C, H) of the ranks before this one, as the all-gather delivers them
    rank_ms, plain_ms, frames = [], [], []
    for r, (f0, f1) in enumerate(frame_split(F, world)):
        last = r == world - 1
        Fr = f1 - f0
        q, k, v = (part(t, f0, f1, N) for t in (x.q, x.k, x.v))
        beta, gamma = part(x.beta, f0, f1, N), part(x.gamma, f0, f1, 1)
        C = torch.empty(B, H, D, D, dtype=torch.float32, device=dev)
        Hc, S_out = torch.empty_like(C), torch.empty_like(C)
        S_buf = [torch.empty_like(C), torch.empty_like(C)]
        o = torch.empty_like(q)
        nb = gdn.gdn_frame_composite_workspace_size(B, H, Fr, N, D)
        ws = torch.empty(nb, dtype=torch.uint8, device=dev)
        prior = list(gathered)

        def start_state():
            S = x.S0
            for i, (Cp, Hp) in enumerate(prior):
                ok(gdn.gdn_state_compose(S, Cp, Hp, S_buf[i % 2], B * H, D, stream), "gdn_state_compose")
                S = S_buf[i % 2]
            return S

        def rank_step():
            ok(gdn.gdn_frame_composite(k, v, beta, gamma, None if last else C, None if last else Hc,
                                       B, H, Fr, N, D, 0.0, ws, nb, stream), "gdn_frame_composite")
            ok(gdn.gdn_frame_fwd_resume(q, gamma, start_state(), S_out, o, B, H, Fr, N, D, ws, nb, stream),
               "gdn_frame_fwd_resume")

        nbf = gdn.gdn_frame_fwd_workspace_size(B, H, Fr, N, D)
        wsf = torch.empty(nbf, dtype=torch.uint8, device=dev)
        of, Sf = torch.empty_like(q), torch.empty_like(C)
        S_plain = start_state()
        S_plain = None if S_plain is None else S_plain.clone()

        def plain_step():
            ok(gdn.gdn_frame_fwd(q, k, v, beta, gamma, S_plain, Sf, of, B, H, Fr, N, D, 0.0, wsf, nbf, stream),
               "gdn_frame_fwd")

        rank_ms.append(timed(rank_step))
        plain_ms.append(timed(plain_step))
        frames.append(Fr)
        if gdn.gdn_device_status() != gdn.GDN_OK:
            raise RuntimeError("device status reports a timed-out wait")
        gathered.append((C.clone(), Hc.clone()))
        del ws, wsf
    return {"ranks": world, "frames": frames, "rank_ms": [round(m, 5) for m in rank_ms],
            "plain_fwd_ms": [round(m, 5) for m in plain_ms],
            "ratio": round(max(a / b for a, b in zip(rank_ms, plain_ms)), 4), "steps": K,
            "note": "ranks run one after another on one GPU; the all-gather between GPUs is not timed"}


def measure_block(x, K, stream, peaks):
    """The GDN block with its projections (gdn_block_fwd) at the layer's shape: x [B, F*N, H*D]
    bf16 with random-init weights W_in [3HD + 2H, HD], W_out [HD, HD]; K calls after 2 warm-ups.
    Also the two projection GEMMs alone, as tensor-pipe throughput against the bf16 peak."""
    import torch
    from gated_deltanet_wise_b300 import gdn
    from gated_deltanet_wise_b300.inputs import make_block_inputs
    B, H, F, N, D = x.B, x.H, x.F, x.N, x.D
    xb = make_block_inputs(B, H, F, N, D, seed=5, device=x.q.device)
    HD, M = H * D, B * F * N
    y = torch.empty_like(xb.x)
    S = torch.empty(B, H, D, D, dtype=torch.float32, device=x.q.device)
    nb = gdn.gdn_block_fwd_workspace_size(B, H, F, N, D)
    ws = torch.empty(nb, dtype=torch.uint8, device=x.q.device)
    q = torch.empty(B, F * N, H, D, dtype=torch.bfloat16, device=x.q.device)
    k, v = torch.empty_like(q), torch.empty_like(q)
    beta = torch.empty(B, F * N, H, device=x.q.device)
    gamma = torch.empty(B, F, H, device=x.q.device)

    def block():
        st = gdn.gdn_block_fwd(xb.x, xb.W_in, xb.W_out, None, S, y, B, H, F, N, D, 0.0, ws, nb, stream)
        if st != gdn.GDN_OK:
            raise gdn.GdnError(st, "gdn_block_fwd")

    def in_proj():
        st = gdn.gdn_block_in_proj(xb.x, xb.W_in, q, k, v, beta, gamma, B, H, F, N, D, stream)
        if st != gdn.GDN_OK:
            raise gdn.GdnError(st, "gdn_block_in_proj")

    def out_proj():
        st = gdn.gdn_block_out_proj(q, xb.W_out, y, B, H, F, N, D, stream)
        if st != gdn.GDN_OK:
            raise gdn.GdnError(st, "gdn_block_out_proj")

    def timed(fn):
        for _ in range(2):
            fn()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0.record(stream)
        for _ in range(K):
            fn()
        t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / K

    ms_block, ms_in, ms_out = timed(block), timed(in_proj), timed(out_proj)
    if gdn.gdn_device_status() != gdn.GDN_OK:
        raise RuntimeError("device status reports a timed-out wait")
    f_in, f_out = 2.0 * M * HD * (3 * HD + 2 * H), 2.0 * M * HD * HD
    sus = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    del ws
    return {"ms_per_step": round(ms_block, 4), "tokens_per_s": round(M / (ms_block * 1e-3), 1),
            "in_proj": {"ms": round(ms_in, 4), "tflops": round(f_in / (ms_in * 1e-3) / 1e12, 1),
                        "tensor_frac": round(f_in / (ms_in * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
                        "tensor_frac_sustained": round(f_in / (ms_in * 1e-3) / 1e12 / sus, 4)},
            "out_proj": {"ms": round(ms_out, 4), "tflops": round(f_out / (ms_out * 1e-3) / 1e12, 1),
                         "tensor_frac": round(f_out / (ms_out * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
                         "tensor_frac_sustained": round(f_out / (ms_out * 1e-3) / 1e12 / sus, 4)},
            "peak_source": ("tensor_frac: bf16_tflops (burst); tensor_frac_sustained: bf16_tflops_sustained "
                            "(a loop of calls runs under the power cap) of MEASURED_PEAKS.json"),
            "steps": K, "gpu_launches_per_step": 7, "d_model": HD}


def measure_backward(x, K, stream, peaks):
    """gdn_frame_bwd on the same layer (dO ~ N(0,1) in bf16, dS_out = 0), K calls after 2 warm-ups.
    Algorithmic bytes: q, k, v, dO read (bf16), beta and gamma read, dq, dk, dv written (fp32),
    dbeta and dgamma written (fp32)."""
    import torch
    from gated_deltanet_wise_b300 import gdn
    B, H, F, N, D = x.B, x.H, x.F, x.N, x.D
    dev = x.q.device
    g = torch.Generator(device=dev).manual_seed(1)
    dO = torch.randn(x.q.shape, generator=g, device=dev).to(torch.bfloat16)
    dq = torch.empty(x.q.shape, dtype=torch.float32, device=dev)
    dk, dv = torch.empty_like(dq), torch.empty_like(dq)
    dbeta = torch.empty(x.beta.shape, dtype=torch.float32, device=dev)
    dgamma = torch.empty(x.gamma.shape, dtype=torch.float32, device=dev)
    dS_in = torch.empty(B, H, D, D, dtype=torch.float32, device=dev)
    nb = gdn.gdn_frame_bwd_workspace_size(B, H, F, N, D)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)

    def step():
        st = gdn.gdn_frame_bwd(x.q, x.k, x.v, x.beta, x.gamma, x.S0, dO, None, dq, dk, dv, dbeta, dgamma, dS_in,
                               B, H, F, N, D, 0.0, ws, nb, stream)
        if st != gdn.GDN_OK:
            raise gdn.GdnError(st, "gdn_frame_bwd")

    for _ in range(2):
        step()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(K):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    if gdn.gdn_device_status() != gdn.GDN_OK:
        raise RuntimeError("device status reports a timed-out wait")
    ms = t0.elapsed_time(t1) / K
    tok = B * F * N * H * D
    alg = 4 * tok * 2 + 3 * tok * 4 + 2 * B * F * N * H * 4 + 2 * B * F * H * 4
    del ws
    return {"ms_per_step": round(ms, 4), "tokens_per_s": round(B * F * N / (ms * 1e-3), 1),
            "algorithmic_bytes": alg, "path_frac_hbm": round(alg / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
            "steps": K, "gpu_launches_per_step": 11, "workspace_bytes": nb}


def run_e2e(x, K, W, world):
    """Same metric through gdn_frame_fwd_host: pinned host inputs -> device -> host outputs, every step."""
    import torch
    from gated_deltanet_wise_b300 import gdn
    B, H, F, N, D = x.B, x.H, x.F, x.N, x.D
    host = {n: getattr(x, n).cpu().pin_memory() for n in ("q", "k", "v", "beta", "gamma")}
    o_h = torch.empty_like(host["q"]).pin_memory()
    S_h = torch.empty(B, H, D, D, dtype=torch.float32).pin_memory()
    nb = gdn.gdn_frame_fwd_host_buffer_size(B, H, F, N, D)
    dbuf = torch.empty(nb, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        st = gdn.gdn_frame_fwd_host(host["q"], host["k"], host["v"], host["beta"], host["gamma"], None, S_h, o_h,
                                    B, H, F, N, D, 0.0, dbuf, nb, stream)
        if st != gdn.GDN_OK:
            raise gdn.GdnError(st, "gdn_frame_fwd_host")

    for _ in range(min(W, 3)):
        step()
    Ke = max(1, min(K, 20))
    torch.cuda.synchronize()
    barrier(world)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(Ke):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = max_over_ranks(world, t0.elapsed_time(t1) / Ke)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = o_h.numel() * o_h.element_size() + S_h.numel() * S_h.element_size()
    return {"value": round(world * B * F * N / (ms * 1e-3), 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 3), "steps": Ke}


# ------------------------------------------------------------- reference arm
def run_reference(args):
    """The fp64 CPU oracle timed on the host cores; each step is a bounded sample of the workload."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    import oracle
    from gated_deltanet_wise_b300.inputs import make_workload
    oracle.build()
    x = make_workload(args.workload, device="cpu", seed=0, F=8)
    threads = oracle.num_threads()
    heads = x.H  # every chain of the layer, as the in-run cpu_baseline samples it
    t1 = oracle_sample(x, heads, 1)
    # size each step to ~2 s so that warm-up + steps finish within a few minutes
    frames = max(1, min(x.F, int(2.0 / max(t1, 1e-3))))
    for _ in range(args.warmup):
        oracle_sample(x, heads, frames)
    ts = [oracle_sample(x, heads, frames) for _ in range(args.steps)]
    t = statistics.fmean(ts)
    tokens_equiv = frames * x.N * heads / x.H
    value = tokens_equiv / t
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "B": 1, "H": 20, "D": 112, "F": 121, "N": 880},
            "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": min(threads, heads),
                             "kind": "oracle",
                             "sample": f"per step: {heads} of 20 heads x {frames} frames x {x.N} tokens, fp64; "
                                       f"scaled to 20-head tokens"},
            "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--frames", type=int, default=None, help="override F (smaller cases for profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-stream", action="store_true", help="skip the streaming-step measurement")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.workload.startswith("streaming"):
        run_streaming_line(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
