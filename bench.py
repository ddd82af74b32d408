"""Benchmark of the dual-mode attention forward pass on GB300.

One step = one pass of the whole hot path (work-list build, the persistent
tcgen05 attention kernel, the split-KV merge) over one batch.  Default
workload: the batch-1 denoise loop (one 256-query bidirectional canvas over a
32768-token cached context, Hq 32 / Hkv 4, head_dim 256); step s uses the
canvas of denoise step s (fresh q and canvas K/V rows, drawn from seed 3+s),
the cached context is reused, as in the loop the method runs.

Timing: W untimed warm-up steps, then K steps.  Before every step (untimed)
the step's canvas rows are written into the resident KV buffer and L2 is
flushed by writing a 256 MiB buffer; each step is timed on its stream with CUDA
events around the call.  ``value`` is algorithmic TFLOP/s (4 * head_dim * Hq *
visible pairs) summed over ranks.  The roofline's kernel time comes from a
second pass over the same K steps with events around the main attention kernel
(events between the call's launches would undo their chaining, so the step
pass has none).  The default run also times the max-throughput mix (full
layer) the same way and reports it under ``configs``.  ``e2e`` times the same steps through the public API with
pinned host buffers: the step's canvas q/k/v go host -> device and out/lse come
back device -> host inside each step's timed interval; the steps are enqueued
back to back, as a serving loop runs them.

``--impl reference`` times the CPU fp64 oracle (the only reference this
method has: there is no code to install) on a bounded sample of the same
workload and prints the same line with ``"impl": "reference"``.
"""

from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from dual_mode_canvas_gb300 import binding  # noqa: E402
from dual_mode_canvas_gb300 import replicas  # noqa: E402
from dual_mode_canvas_gb300 import workloads as wls  # noqa: E402

METRIC = "dual-mode attention TFLOP/s and denoise steps/s; % of tensor/HBM roofline"
L2_FLUSH_BYTES = 256 << 20
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def visible_pairs(wl) -> int:
    """Visible (query, key) pairs of one query head: sum over rows of the
    window size clipped to the sequence (causal: j <= i, bidirectional: all
    keys; W narrows both)."""
    tot = 0
    W = wl.window
    for c, n, md in wl.seqs:
        L = c + n
        i = c + np.arange(n, dtype=np.int64)
        lo = np.zeros_like(i) if W < 0 else np.maximum(0, i - W)
        if md == wls.CAUSAL:
            hi = i
        else:
            hi = np.full_like(i, L - 1) if W < 0 else np.minimum(L - 1, i + W)
        tot += int((hi - lo + 1).sum())
    return tot


def algorithmic_flops(wl) -> int:
    return 4 * wl.head_dim * wl.num_q_heads * visible_pairs(wl)


def algorithmic_bytes(wl, qkv_bytes: int = 2) -> int:
    """Q + out (bf16) + lse (fp32) + every K/V row some query sees, read once per KV head
    (Q, K, V of ``qkv_bytes`` per element: 2 for bf16, 1 for e4m3)."""
    W = wl.window
    kv = 0
    for c, n, md in wl.seqs:
        L = c + n
        lo = 0 if W < 0 else max(0, c - W)
        hi = c + n - 1 if md == wls.CAUSAL else (L - 1 if W < 0 else min(L - 1, c + n - 1 + W))
        kv += hi - lo + 1
    q = wl.total_q * wl.num_q_heads * wl.head_dim
    return (q * qkv_bytes + q * 2 + wl.total_q * wl.num_q_heads * 4 +
            2 * kv * wl.num_kv_heads * wl.head_dim * qkv_bytes)


def load_peaks():
    if os.path.exists(PEAKS_FILE):
        with open(PEAKS_FILE) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


class ClockSampler:
    """SM clock and clock-event-reason sampling during the timed region.

    Polls NVML (read-only queries through ctypes) from a background thread
    every ~0.5 ms, so even a few-millisecond timed region is covered; falls
    back to ``nvidia-smi -lms 100`` when NVML cannot be loaded."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int):
        self.dev = device_index
        self.samples = []
        self.max_mhz = None
        self._stop = False
        self._thread = None
        self._nvml = None
        self._handle = None
        self.source = "none"

    def _open_nvml(self):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return False
        if lib.nvmlInit_v2() != 0:
            return False
        handle = ctypes.c_void_p()
        try:
            bus = torch.cuda.get_device_properties(self.dev)
            busid = f"{bus.pci_domain_id:08x}:{bus.pci_bus_id:02x}:{bus.pci_device_id:02x}.0".encode()
            rc = lib.nvmlDeviceGetHandleByPciBusId_v2(busid, ctypes.byref(handle))
        except AttributeError:
            rc = 1
        if rc != 0 and lib.nvmlDeviceGetHandleByIndex_v2(self.dev, ctypes.byref(handle)) != 0:
            return False
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        self._nvml, self._handle = lib, handle
        return True

    def _poll(self):
        import ctypes
        mhz, reasons = ctypes.c_uint(), ctypes.c_ulonglong()
        get_reasons = getattr(self._nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self._nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop:
            if self._nvml.nvmlDeviceGetClockInfo(self._handle, 1, ctypes.byref(mhz)) == 0:
                rs = reasons.value if get_reasons(self._handle, ctypes.byref(reasons)) == 0 else 0
                self.samples.append((float(mhz.value), int(rs)))
            time.sleep(0.0005)

    def __enter__(self):
        import threading
        if self._open_nvml():
            self.source = "nvml"
            self._thread = threading.Thread(target=self._poll, daemon=True)
            self._thread.start()
            t0 = time.perf_counter()
            while not self.samples and time.perf_counter() - t0 < 1.0:
                time.sleep(0.001)
        else:
            self.source = "nvidia-smi"
            self._proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), "--query-gpu=clocks.sm,clocks.max.sm",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop = True
            self._thread.join(timeout=5)
        elif self.source == "nvidia-smi":
            self._proc.terminate()
            out, _ = self._proc.communicate(timeout=10)
            for ln in out.splitlines():
                parts = [x.strip() for x in ln.split(",")]
                try:
                    self.samples.append((float(parts[0]), 0))
                    self.max_mhz = float(parts[1])
                except (ValueError, IndexError):
                    pass

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unsampled"],
                    "samples": 0, "source": self.source}
        reasons = set()
        for _, rs in self.samples:
            for bit, name in self.REASONS.items():
                if rs & bit:
                    reasons.add(name)
        return {"sm_mhz": float(np.median([m for m, _ in self.samples])), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(self.samples), "source": self.source}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    replicas.barrier()


def max_over_ranks(world, x: float) -> float:
    return replicas.aggregate(x, 0.0, device="cuda")[0]


def measure_attention(wl, args, world, local, page_size=0, fp8=False):
    """W warm-up and K timed steps of one attention workload on this rank.
    Returns the per-step and per-kernel times (max over ranks), the clock
    record of the timed region and, for the denoise loop, the end-to-end
    record through the public API with host buffers."""
    dev = torch.device("cuda")
    paged = page_size > 0
    if fp8:
        # e4m3 codes with one scale per tensor; later canvases use step 0's scales
        batch = wls.make_fp8_batch(wl, device="cuda")
        q, k, v = batch["q8"], batch["k8"], batch["v8"]
        sc8 = (batch["q_scale"], batch["k_scale"], batch["v_scale"])
        rows = wls.canvas_rows(wl)
    elif paged:
        # paged KV cache: the step's canvas K/V go in as k_new / v_new and the
        # call appends them into their pages (inside the timed call)
        batch = wls.make_paged_batch(wl, page_size, device="cuda")
        q, k, v = batch["q"], batch["k_new"], batch["v_new"]
        k_cache, v_cache = batch["k_cache"], batch["v_cache"]
        bt = batch["block_table"].cuda()
        rows = [(0, wl.total_q)]  # k / v here are the new rows themselves
    else:
        batch = wls.make_batch(wl, device="cuda")
        q, k, v = batch["q"], batch["k"], batch["v"]
        rows = wls.canvas_rows(wl)
    cu_q, ctx, mode = batch["cu_q"].cuda(), batch["ctx_len"].cuda(), batch["mode"].cuda()
    nsteps = args.warmup + args.steps
    loop = wl.steps > 1
    # canvases of every step, drawn up front (device) and mirrored in pinned host memory
    canv = []
    if loop:
        for s in range(nsteps):
            step = s % wl.steps
            if step == 0:
                qs = q.clone()
                kc = torch.cat([k[a:b] for a, b in rows])
                vc = torch.cat([v[a:b] for a, b in rows])
            else:
                qs, kc, vc = wls.denoise_step_inputs(wl, step, device="cuda")
                if fp8:
                    qs = wls.quantize_e4m3(qs.float(), sc8[0])
                    kc = wls.quantize_e4m3(kc.float(), sc8[1])
                    vc = wls.quantize_e4m3(vc.float(), sc8[2])
            canv.append((qs, kc, vc))
    out = torch.empty((wl.total_q, wl.num_q_heads, wl.head_dim), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((wl.total_q, wl.num_q_heads), dtype=torch.float32, device=dev)
    ws = torch.empty(binding.workspace_size(len(wl.seqs), wl.total_q, wl.num_q_heads,
                                            wl.num_kv_heads, wl.head_dim), dtype=torch.uint8,
                     device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def stage(s):
        if loop:
            qs, kc, vc = canv[s]
            q.copy_(qs)
            o = 0
            for a, b in rows:
                k[a:b].copy_(kc[o:o + b - a])
                v[a:b].copy_(vc[o:o + b - a])
                o += b - a
        flush.fill_(s & 0xFF)

    def call(events=None):
        if fp8:
            binding.forward_fp8(q, k, v, cu_q, ctx, mode, wl.window, wl.scale, *sc8, out=out, lse=lse,
                                workspace=ws, events=events)
        elif paged:
            binding.forward_paged(q, k, v, k_cache, v_cache, bt, cu_q, ctx, mode, wl.window, wl.scale,
                                  out=out, lse=lse, workspace=ws, events=events)
        else:
            binding.forward(q, k, v, cu_q, ctx, mode, wl.window, wl.scale, out=out, lse=lse,
                            workspace=ws, events=events)

    flops = algorithmic_flops(wl)
    nbytes = algorithmic_bytes(wl, 1 if fp8 else 2)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(nsteps)]
    for e in ev:  # torch creates CUDA events lazily, on their first record
        for x in e:
            x.record(stream)
    for s in range(args.warmup):
        stage(s)
        call()
    torch.cuda.synchronize()
    st = binding.status()
    if st != binding.DG_OK:
        raise RuntimeError(f"device status {st}: {binding.error_string(st)}")

    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    torch.cuda.nvtx.range_push("timed steps")
    with ClockSampler(local) as clk:
        # the steps as a caller runs them: events only around each call, so the
        # call's three launches stay chained as programmatic dependents
        for s in range(args.warmup, nsteps):
            stage(s)
            e0, e1, _, _ = ev[s]
            e0.record(stream)
            call()
            e1.record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall0
        # the same steps again with events around the main kernel alone (they
        # sit between the launches and undo the chaining, so this pass gives
        # the kernel time, not the step time)
        for s in range(args.warmup, nsteps):
            stage(s)
            _, _, a0, a1 = ev[s]
            call(events=(a0, a1))
        torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    barrier(world)
    st = binding.status()
    if st != binding.DG_OK:
        raise RuntimeError(f"device status {st}: {binding.error_string(st)}")
    step_ms = [ev[s][0].elapsed_time(ev[s][1]) for s in range(args.warmup, nsteps)]
    attn_ms = [ev[s][2].elapsed_time(ev[s][3]) for s in range(args.warmup, nsteps)]
    tot_ms = max_over_ranks(world, float(sum(step_ms)))
    ms_per_step = tot_ms / args.steps
    attn_avg_ms = max_over_ranks(world, float(np.mean(attn_ms)))

    # ---------------------------------------------- end to end, host buffers
    e2e = None
    if loop:
        hq = [c[0].cpu().pin_memory() for c in canv]
        hk = [c[1].cpu().pin_memory() for c in canv]
        hv = [c[2].cpu().pin_memory() for c in canv]
        esz = hq[0].element_size()
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        # steps are enqueued back to back (as a serving loop runs them); each
        # is timed on the device between its events.  The canvas K/V rows go
        # from pinned host memory straight into their rows of the KV buffer.
        ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(nsteps)]
        for s in range(nsteps):
            flush.fill_(s & 0xFF)
            e0, e1 = ev2[s]
            e0.record(stream)
            q.copy_(hq[s], non_blocking=True)
            o = 0
            for a, b in rows:
                k[a:b].copy_(hk[s][o:o + b - a], non_blocking=True)
                v[a:b].copy_(hv[s][o:o + b - a], non_blocking=True)
                o += b - a
            call()
            h_out.copy_(out, non_blocking=True)
            h_lse.copy_(lse, non_blocking=True)
            e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = [ev2[s][0].elapsed_time(ev2[s][1]) for s in range(args.warmup, nsteps)]
        e2e_tot = max_over_ranks(world, float(sum(e2e_ms)))
        h2d = (hq[0].numel() + hk[0].numel() + hv[0].numel()) * esz
        d2h = h_out.numel() * 2 + h_lse.numel() * 4
        e2e = {"value": world * flops * args.steps / (e2e_tot * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_tot / args.steps}

    return {"wl": wl, "flops": flops, "nbytes": nbytes, "tot_ms": tot_ms, "ms_per_step": ms_per_step,
            "attn_avg_ms": attn_avg_ms, "t_wall": t_wall, "clocks": clk.summary(), "e2e": e2e,
            "steps": args.steps, "paged": paged, "fp8": fp8}


def source_sha16():
    """Hash of the attention kernel's sources (device code and the host code
    that chooses its shapes and launch)."""
    import hashlib
    h = hashlib.sha256()
    for f in ("kernels.cuh", "ptx.cuh", "dg_attn.cu"):
        with open(os.path.join(ROOT, "dual_mode_canvas_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(key):
    """dram__bytes_read.sum + dram__bytes_write.sum of one main-kernel launch of
    workload ``key`` from the ncu capture listed in profiles/traffic_bytes.txt,
    or None when that capture was taken of other kernel sources than these."""
    path = os.path.join(ROOT, "profiles", "traffic_bytes.txt")
    if not os.path.exists(path):
        return None
    sha = source_sha16()
    with open(path) as f:
        for ln in f:
            parts = ln.split("#")[0].split()
            if len(parts) == 3 and parts[0] == key and parts[1] == sha:
                return float(parts[2])
    return None


def attention_roofline(m, peaks, peaks_src, key):
    """Roofline record of the main attention kernel from a measurement."""
    flops, nbytes, attn_avg_ms = m["flops"], m["nbytes"], m["attn_avg_ms"]
    attn_tflops = flops / (attn_avg_ms * 1e-3) / 1e12
    sustained = m["steps"] * m["ms_per_step"] > 1000.0
    tc_peak = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
    if m["fp8"]:
        tc_peak = tc_peak * 2.0  # the nominal e4m3 / bf16 dense ratio (4.5 / 2.25 PFLOP/s)
    t_tc = flops / (tc_peak * 1e12)
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    bound = "tensor" if t_tc >= t_hbm else "hbm"
    if bound == "tensor":
        roof = {"bound": "tensor", "achieved": round(attn_tflops, 2), "peak": tc_peak,
                "unit": "TFLOP/s", "frac": round(attn_tflops / tc_peak, 4)}
    else:
        gbs = nbytes / (attn_avg_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(gbs / peaks["hbm_gbs"], 4)}
    roof["traffic"] = None if m["paged"] else ncu_traffic(key)
    roof["traffic_source"] = ("ncu capture of these kernel sources (profiles/traffic_bytes.txt)"
                              if roof["traffic"] is not None else
                              "none for these kernel sources (sha " + source_sha16() + ")")
    roof["peak_source"] = f"{peaks_src} ({'sustained' if (sustained and bound == 'tensor') else 'burst'})" + (
        "; e4m3 peak = measured bf16 x 2 (nominal ratio)" if m["fp8"] else "")
    roof["kernel"] = "fwd_kernel (persistent tcgen05 attention)"
    roof["kernel_ms_per_launch"] = round(attn_avg_ms, 4)
    roof["tighter_roof_frac"] = round(max(t_tc, t_hbm) / (attn_avg_ms * 1e-3), 4)
    return roof


def run_gpu(args):
    world, rank, local = dist_setup()
    binding.load_library()
    paged = args.paged > 0
    fp8 = args.fp8
    if fp8 and paged:
        raise SystemExit("--fp8 runs on the contiguous layout only")
    wl = wls.WORKLOADS[args.workload]
    m = measure_attention(wl, args, world, local, args.paged, fp8)
    # the second graded configuration (the max-throughput mix, full layer)
    # is timed in the same run, after the headline workload
    m4 = None
    if args.workload == "denoise_loop" and not paged and not fp8 and not args.headline_only:
        m4 = measure_attention(wls.WORKLOADS["maxmix_full"], args, world, local)
    if rank != 0:
        return
    peaks, peaks_src = load_peaks()
    key = args.workload + (":e4m3" if fp8 else "")
    tot_ms, ms_per_step, flops, nbytes = m["tot_ms"], m["ms_per_step"], m["flops"], m["nbytes"]
    tflops = world * flops * args.steps / (tot_ms * 1e-3) / 1e12
    roof = attention_roofline(m, peaks, peaks_src, key)
    e2e, t_wall, clk = m["e2e"], m["t_wall"], m["clocks"]
    res = {
        "metric": METRIC, "value": round(tflops, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if fp8 else "bf16",
        "data": "synthetic (seeded N(0,1), e4m3 with one scale per tensor)" if fp8 else
                "synthetic (seeded N(0,1), bf16)",
        "config": {"workload": wl.name, "seqs_ctx_nq_mode": [list(s) for s in wl.seqs],
                   "num_q_heads": wl.num_q_heads, "num_kv_heads": wl.num_kv_heads,
                   "head_dim": wl.head_dim, "window": wl.window,
                   "l2": "flushed before every step (256 MiB write)",
                   "kv_layout": (f"paged: {args.paged}-row pages, shuffled page table, canvas K/V "
                                 "appended inside the timed call") if paged else "contiguous",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "denoise_steps_per_s": round(1000.0 / ms_per_step, 2),
        "algorithmic_gflop_per_step": round(flops / 1e9, 3),
        "algorithmic_mb_per_step": round(nbytes / 1e6, 3),
        "wall_s_timed_region": round(t_wall, 3),
        "gpu_launches": binding.launches_per_call(len(wl.seqs), wl.total_q, wl.num_q_heads, wl.num_kv_heads,
                                                  wl.head_dim, paged, fp8) * args.steps * world,
        "roofline": roof,
        "clocks": clk,
    }
    if m4 is not None:
        w4 = m4["wl"]
        res["configs"] = {"maxmix_full": {
            "workload": w4.name, "seqs_ctx_nq_mode": [list(x) for x in w4.seqs],
            "num_q_heads": w4.num_q_heads, "num_kv_heads": w4.num_kv_heads, "head_dim": w4.head_dim,
            "window": w4.window, "steps": args.steps, "warmup": args.warmup,
            "value": round(world * m4["flops"] * args.steps / (m4["tot_ms"] * 1e-3) / 1e12, 2),
            "unit": "TFLOP/s", "ms_per_step": round(m4["ms_per_step"], 4),
            "algorithmic_gflop_per_step": round(m4["flops"] / 1e9, 3),
            "algorithmic_mb_per_step": round(m4["nbytes"] / 1e6, 3),
            "l2": "flushed before every step (256 MiB write)",
            "gpu_launches": binding.launches_per_call(len(w4.seqs), w4.total_q, w4.num_q_heads,
                                                      w4.num_kv_heads, w4.head_dim) * args.steps * world,
            "roofline": attention_roofline(m4, peaks, peaks_src, "maxmix_full"),
            "clocks": m4["clocks"]}}
    if e2e is not None:
        res["e2e"] = e2e
    if not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(wl, budget_s=args.cpu_seconds)
    print(json.dumps(res))


def _oracle_sample(wl, q_heads):
    """The bounded CPU sample: the first sequence's queries, ``q_heads`` query
    heads of KV head 0, against its KV rows, through the fp64 oracle."""
    import oracle
    batch = wls.make_batch(wl, device="cpu") if wl.total_kv < (1 << 16) else None
    if batch is None:
        # build just the first sequence's rows on the host (same generator recipe)
        b = wls.make_batch(wl, device="cuda")
        c, n, md = wl.seqs[0]
        qs = b["q"][:n, :q_heads].float().cpu().numpy().astype(np.float64)
        ks = b["k"][:c + n, :1].float().cpu().numpy().astype(np.float64)
        vs = b["v"][:c + n, :1].float().cpu().numpy().astype(np.float64)
    else:
        c, n, md = wl.seqs[0]
        qs = batch["q"][:n, :q_heads].float().numpy().astype(np.float64)
        ks = batch["k"][:c + n, :1].float().numpy().astype(np.float64)
        vs = batch["v"][:c + n, :1].float().numpy().astype(np.float64)
    one = wls.Workload("sample", (wl.seqs[0],), q_heads, 1, wl.head_dim, wl.window, wl.seed)
    flops = algorithmic_flops(one)

    def run():
        oracle.attention(qs, ks, vs, [0, n], [c], [md], wl.window, wl.scale)
    return run, flops


def cpu_baseline(wl, budget_s=15.0):
    heads = max(1, wl.num_q_heads // wl.num_kv_heads)
    run, flops = _oracle_sample(wl, heads)
    t0 = time.perf_counter()
    reps = 0
    while True:
        run()
        reps += 1
        if time.perf_counter() - t0 > budget_s or reps >= 50:
            break
    dt = time.perf_counter() - t0
    return {"value": round(flops * reps / dt / 1e12, 6), "unit": "TFLOP/s",
            "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"fp64 NumPy oracle, first sequence of {wl.name}, {heads} query heads of KV head 0 "
                      f"(of {wl.num_q_heads}), {reps} repetition(s) in {dt:.1f} s"}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    wl = wls.WORKLOADS[args.workload]
    run, flops = _oracle_sample(wl, 1)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = time.perf_counter() - t0
    val = flops * args.steps / dt / 1e12
    res = {"impl": "reference", "metric": METRIC, "value": round(val, 6), "unit": "TFLOP/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1), bf16)",
           "config": {"workload": wl.name, "sample": "first sequence, 1 query head"},
           "cpu_baseline": {"value": round(val, 6), "unit": "TFLOP/s", "kind": "oracle",
                            "cores": len(os.sched_getaffinity(0)),
                            "sample": f"fp64 NumPy oracle, first sequence of {wl.name}, query head 0 "
                                      f"per step"},
           "e2e": {"value": round(val, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(res))


def run_accept(args):
    """The entropy-bounded acceptance step of one denoise step (HBM-bound: one
    pass over the LM-head logits).  Value: logits bytes / kernel time."""
    world, rank, local = dist_setup()
    wl = wls.LOGITS_WORKLOADS[args.workload]
    binding.load_library()
    x, cu = wls.make_logits(wl, device="cuda")
    cu = cu.cuda()
    rows = wl.rows
    acc_in = torch.zeros(rows, dtype=torch.uint8, device="cuda")
    prev = torch.zeros(rows, dtype=torch.int32, device="cuda")
    stable = torch.zeros(len(wl.canvases), dtype=torch.int32, device="cuda")
    ws = torch.empty(binding.load_library().dg_accept_workspace_size(rows, wl.vocab),
                     dtype=torch.uint8, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    nsteps = args.warmup + args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(nsteps)]
    stream = torch.cuda.current_stream()
    for s_ in range(args.warmup):
        flush.fill_(s_ & 0xFF)
        binding.accept_step(x, cu, acc_in, prev, stable, 2.0, 3.0, 3, s_, 48, workspace=ws,
                            events=ev[s_])
    torch.cuda.synchronize()
    barrier(world)
    with ClockSampler(local) as clk:
        for s_ in range(args.warmup, nsteps):
            flush.fill_(s_ & 0xFF)
            binding.accept_step(x, cu, acc_in, prev, stable, 2.0, 3.0, 3, s_, 48, workspace=ws,
                                events=ev[s_])
        torch.cuda.synchronize()
    barrier(world)
    st = binding.status()
    if st != binding.DG_OK:
        raise RuntimeError(f"device status {st}")
    ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(args.warmup, nsteps)]
    tot = max_over_ranks(world, float(sum(ms)))
    nbytes = x.numel() * 2 + rows * (4 + 4 + 4 + 1 + 1 + 4)

    # end to end: the step's logits host -> device, the per-row results and
    # per-canvas flags device -> host
    hx = x.cpu().pin_memory()
    res_h = None
    ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(nsteps)]
    for s_ in range(nsteps):  # enqueued back to back, each step timed between its events
        flush.fill_(s_ & 0xFF)
        e0, e1 = ev2[s_]
        e0.record(stream)
        x.copy_(hx, non_blocking=True)
        res = binding.accept_step(x, cu, acc_in, prev, stable, 2.0, 3.0, 3, s_, 48, workspace=ws)
        res_h = {k: v.to("cpu", non_blocking=True) for k, v in res.items()}
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = [ev2[i][0].elapsed_time(ev2[i][1]) for i in range(args.warmup, nsteps)]
    e2e_tot = max_over_ranks(world, float(sum(e2e_ms)))
    d2h = sum(v.numel() * v.element_size() for v in res_h.values())
    if rank != 0:
        return
    peaks, src = load_peaks()
    gbs = world * nbytes * args.steps / (tot * 1e-3) / 1e9
    kgbs = nbytes / (float(np.mean(ms)) * 1e-3) / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        import oracle.acceptance as oacc
        sample = x[:8].float().cpu().numpy()
        t0 = time.perf_counter()
        reps = 0
        while time.perf_counter() - t0 < args.cpu_seconds and reps < 50:
            oacc.row_stats(sample)
            reps += 1
        dt = time.perf_counter() - t0
        cpu = {"value": round(sample.size * 2 * reps / dt / 1e9, 3), "unit": "GB/s",
               "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
               "sample": f"fp64 NumPy oracle row statistics of 8 of {rows} rows x {wl.vocab} "
                         f"logits, {reps} repetition(s) in {dt:.1f} s (bf16 bytes counted)"}
    line = {
        "metric": "entropy-bounded acceptance step GB/s (logits read once)", "value": round(gbs, 1),
        "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot / args.steps, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded logits, bf16)",
        "config": {"workload": wl.name, "canvases": list(wl.canvases), "vocab": wl.vocab,
                   "l2": "flushed before every step (256 MiB write)"},
        "gpu_launches": 2 * args.steps * world,
        "roofline": {"bound": "hbm", "achieved": round(kgbs, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(kgbs / peaks["hbm_gbs"], 4), "traffic": None,
                     "peak_source": src, "kernel": "row_stats_kernel + accept_kernel"},
        "clocks": clk.summary(),
        "e2e": {"value": round(world * nbytes * args.steps / (e2e_tot * 1e-3) / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": x.numel() * 2, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_tot / args.steps, 4)}}
    if cpu is not None:
        line["cpu_baseline"] = cpu
    print(json.dumps(line))


def _a256(n):
    return (n + 255) // 256 * 256


def run_selfcond(args):
    """The self-conditioning embedding average of one denoise step: softmax of
    the LM-head logits times the token-embedding table (tensor-bound).  Value:
    2 * rows * vocab * d_model / step time."""
    world, rank, local = dist_setup()
    wl = wls.SELFCOND_WORKLOADS[args.workload]
    binding.load_library()
    x, _ = wls.make_logits(wl.logits, device="cuda")
    E = wls.make_embedding(wl.logits.vocab, wl.d_model, wl.seed, device="cuda")
    rows, vocab, d = wl.logits.rows, wl.logits.vocab, wl.d_model
    out = torch.empty((rows, d), dtype=torch.float32, device="cuda")
    lib = binding.load_library()
    ws = torch.empty(lib.dg_sampler_workspace_size(rows, vocab, d) if args.sampler
                     else lib.dg_selfcond_workspace_size(rows, vocab, d), dtype=torch.uint8, device="cuda")
    if args.sampler:
        # the whole sampler step: acceptance and self-conditioning sharing one
        # pass of row statistics
        _, cu_rows = wls.make_logits(wl.logits, device="cpu")
        cu_rows = cu_rows.cuda()
        acc_in = torch.zeros(rows, dtype=torch.uint8, device="cuda")
        prev = torch.zeros(rows, dtype=torch.int32, device="cuda")
        stab = torch.zeros(len(wl.logits.canvases), dtype=torch.int32, device="cuda")

    def sc_call(events=None):
        """One step; returns the self-conditioning output tensor."""
        if args.sampler:
            return binding.sampler_step(x, cu_rows, acc_in, prev, stab, 2.0, 3.0, 3, 0, 48, E,
                                        workspace=ws, events=events)["selfcond"]
        return binding.self_conditioning(x, E, out=out, workspace=ws, events=events)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    nsteps = args.warmup + args.steps
    ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(4)) for _ in range(nsteps)]
    for e in ev:
        for y in e:
            y.record(stream)
    for s_ in range(args.warmup):
        flush.fill_(s_ & 0xFF)
        sc_call()
    torch.cuda.synchronize()
    barrier(world)
    with ClockSampler(local) as clk:
        for s_ in range(args.warmup, nsteps):
            flush.fill_(s_ & 0xFF)
            e0, e1, a0, a1 = ev[s_]
            e0.record(stream)
            sc_call(events=(a0, a1))
            e1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    st = binding.status()
    if st != binding.DG_OK:
        raise RuntimeError(f"device status {st}")
    ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(args.warmup, nsteps)]
    kms = [ev[i][2].elapsed_time(ev[i][3]) for i in range(args.warmup, nsteps)]
    tot = max_over_ranks(world, float(sum(ms)))
    kavg = max_over_ranks(world, float(np.mean(kms)))
    flops = 2.0 * rows * vocab * d
    nbytes = x.numel() * 2 + E.numel() * 2 + out.numel() * 4

    # end to end: the step's logits host -> device, the result device -> host
    hx = x.cpu().pin_memory()
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(nsteps)]
    for s_ in range(nsteps):  # enqueued back to back, each step timed between its events
        flush.fill_(s_ & 0xFF)
        e0, e1 = ev2[s_]
        e0.record(stream)
        x.copy_(hx, non_blocking=True)
        h_out.copy_(sc_call(), non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = [ev2[i][0].elapsed_time(ev2[i][1]) for i in range(args.warmup, nsteps)]
    e2e_tot = max_over_ranks(world, float(sum(e2e_ms)))
    if rank != 0:
        return
    peaks, src = load_peaks()
    sustained = tot > 1000.0
    tc_peak = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
    tflops = world * flops * args.steps / (tot * 1e-3) / 1e12
    ktf = flops / (kavg * 1e-3) / 1e12
    t_tc = flops / (tc_peak * 1e12)
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    res = {
        "metric": "self-conditioning embedding average TFLOP/s (softmax(logits) x E)",
        "value": round(tflops, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(tot / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded logits and N(0,1) embeddings, bf16)",
        "config": {"workload": wl.name + ("+acceptance (dg_sampler_step)" if args.sampler else ""),
                   "rows": rows, "vocab": vocab, "d_model": d,
                   "l2": "flushed before every step (256 MiB write)"},
        # row statistics, row constants, the GEMM, and the split sum when the
        # workspace holds per-split partials (beyond the statistics)
        "gpu_launches": ((4 if ws.numel() > _a256(16 * rows * -(-(vocab + (7 if vocab % 8 else 0)) // 16384))
                          + _a256(4 * rows) else 3) + (1 if args.sampler else 0)) * args.steps * world,
        "roofline": {"bound": "tensor" if t_tc >= t_hbm else "hbm", "achieved": round(ktf, 2),
                     "peak": tc_peak, "unit": "TFLOP/s", "frac": round(ktf / tc_peak, 4),
                     "traffic": None,
                     "peak_source": f"{src} ({'sustained' if sustained else 'burst'})",
                     "kernel": ("dg_sampler_step, whole call (events around the call)" if args.sampler
                                else "sc_kernel (persistent tcgen05 softmax x E)"),
                     "kernel_ms_per_launch": round(kavg, 4),
                     "tighter_roof_frac": round(max(t_tc, t_hbm) / (kavg * 1e-3), 4)},
        "clocks": clk.summary(),
        "e2e": {"value": round(world * flops * args.steps / (e2e_tot * 1e-3) / 1e12, 2),
                "unit": "TFLOP/s", "h2d_bytes_per_step": x.numel() * 2,
                "d2h_bytes_per_step": out.numel() * 4, "ms_per_step": round(e2e_tot / args.steps, 4)},
    }
    if not args.no_cpu_baseline:
        import oracle.selfcond as sc
        xr = x[:2].float().cpu().numpy().astype(np.float64)
        Ec = E[:, :256].float().cpu().numpy().astype(np.float64)
        t0 = time.perf_counter()
        reps = 0
        while time.perf_counter() - t0 < args.cpu_seconds and reps < 50:
            sc.self_conditioning(xr, Ec)
            reps += 1
        dt = time.perf_counter() - t0
        res["cpu_baseline"] = {"value": round(2.0 * 2 * vocab * 256 * reps / dt / 1e12, 6),
                               "unit": "TFLOP/s", "cores": len(os.sched_getaffinity(0)),
                               "kind": "oracle",
                               "sample": f"fp64 NumPy oracle, 2 rows x {vocab} vocabulary x 256 of {d} "
                                         f"columns, {reps} repetition(s) in {dt:.1f} s"}
    print(json.dumps(res))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--fp8", action="store_true",
                    help="run the attention in e4m3 (Q, K, V codes with one scale per tensor)")
    ap.add_argument("--sampler", action="store_true",
                    help="self-conditioning workloads: time the combined sampler step (acceptance + "
                         "self-conditioning sharing one statistics pass)")
    ap.add_argument("--paged", type=int, default=0,
                    help="page size: run the step through the paged KV cache (0: contiguous)")
    ap.add_argument("--workload", default="denoise_loop",
                    choices=sorted(wls.WORKLOADS) + sorted(wls.LOGITS_WORKLOADS) +
                    sorted(wls.SELFCOND_WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true",
                    help="time only the chosen workload (the default run also times the max-throughput "
                         "mix, full layer, as a nested record)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "gb300":
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus != world:
        # one process per GPU: N GPUs need N ranks from a launcher
        ap.error(f"--gpus {args.gpus} needs {args.gpus} ranks (python -m torch.distributed.run "
                 f"--nproc-per-node {args.gpus} bench.py --gpus {args.gpus} ...); this process "
                 f"sees WORLD_SIZE={world}")
    if args.impl == "reference":
        run_reference(args)
    elif args.workload in wls.LOGITS_WORKLOADS:
        run_accept(args)
    elif args.workload in wls.SELFCOND_WORKLOADS:
        run_selfcond(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
