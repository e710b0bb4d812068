#!/usr/bin/env python
"""MLA decode benchmark on GB300: one JSON line on rank 0.

A step is one pass of the whole decode hot path (scheduler metadata, split
kernel, combine: its own kernel, or the split kernel's fused phase when the
schedule splits no sequence) over one batch of the chosen synthetic workload
(default: paged bf16, b=64, h=128, cache 4096, 64-token pages, shuffled block
table).  Inputs are resident in HBM; the step rotates over several input sets
whose KV caches are each larger than the 129 MB L2.  `value` is TFLOP/s with
flops counted as b*h*sum(L)*2*(576+512); the effective HBM bandwidth, the
roofline of the split kernel, an end-to-end figure through the public API with
host buffers, clock samples and the oracle's CPU baseline ride along.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs an independent replica (weak scaling; no
collective on the data path: only a barrier and a max-reduction of times).
"""
import argparse
import ctypes
import glob
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("MLA decode TFLOPS and effective HBM GB/s on 1 GB300 (paged bf16), "
          "% of roofline")
UNIT = "TFLOP/s"
FALLBACK_HBM_GBS = 6800.0
EVENT_EVERY = 10  # timed steps between two event-instrumented split launches
PREQUEUE_CYCLES = 1_000_000  # ~0.5 ms of SM clocks of device-side delay before the timed region
FALLBACK_BF16_TFLOPS = 1900.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="paged")
    ap.add_argument("--copies", type=int, default=3, help="rotating input sets (L2 defeat)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch (smaller cases for profiler captures)")
    ap.add_argument("--layout", choices=["fused", "split"], default="fused",
                    help="fused: 576-column q / kv_cache rows; split: Q / Q_pe and KV / K_pe "
                         "as separate tensors")
    ap.add_argument("--combine", choices=["auto", "fused", "kernel"], default="auto",
                    help="fused: the split kernel combines the sequences it split (grid "
                         "barrier); kernel: a separate combine kernel after it; auto: "
                         "fused when the schedule splits no sequence (no combine then "
                         "runs at all), else the combine kernel, decided once from the "
                         "batch's metadata before anything is timed")
    return ap.parse_args()


def as_layout(s, layout):
    """The decode tensors of input set `s` in the chosen layout (q_pe / k_pe None when fused)."""
    d = dict(s, q_pe=None, k_pe=None)
    if layout == "split":
        q, kv = s["q"], s["kv_cache"]
        d.update(q=q[..., :512].contiguous(), q_pe=q[..., 512:].contiguous(),
                 kv_cache=kv[..., :512].contiguous(), k_pe=kv[..., 512:].contiguous())
    return d


# ------------------------------------------------------------------------------- helpers

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def kernel_source_hash():
    """Hash of the split kernel's sources (the kernel the roofline line reports)."""
    csrc = os.path.join(ROOT, "mla_decode_gb300", "csrc")
    files = [os.path.join(csrc, f) for f in ("combine.cuh", "common.cuh", "internal.h", "sm100.cuh",
                                             "split_sm103.cu")]
    h = hashlib.sha256()
    for f in files:
        h.update(os.path.basename(f).encode())
        h.update(open(f, "rb").read())
    return h.hexdigest()[:12]


def ncu_traffic(workload):
    """DRAM bytes per split-kernel launch from a committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    want = kernel_source_hash()
    for path in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        kv = {}
        for line in open(path):
            if ":" in line and line.startswith("- "):
                k, v = line[2:].split(":", 1)
                kv[k.strip()] = v.strip().strip("`")
        if (kv.get("kernel") == "split" and kv.get("workload") == workload
                and kv.get("source_hash") == want and "traffic_bytes_per_launch" in kv):
            try:
                return float(kv["traffic_bytes_per_launch"])
            except ValueError:
                return None
    return None


class ClockSampler:
    """Samples SM clock and clock-event reasons while the timed region runs (NVML via
    ctypes, falling back to nvidia-smi)."""
    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}

    def __init__(self, torch_index):
        self.samples = []
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._proc = None
        self.nvml = None
        try:
            import torch
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            handle = ctypes.c_void_p()
            props = torch.cuda.get_device_properties(torch_index)
            uuid = getattr(props, "uuid", None)
            ok = False
            if uuid is not None:
                s = str(uuid)
                s = s if s.startswith("GPU-") else "GPU-" + s
                ok = lib.nvmlDeviceGetHandleByUUID(s.encode(), ctypes.byref(handle)) == 0
            if not ok:
                ok = lib.nvmlDeviceGetHandleByIndex_v2(torch_index, ctypes.byref(handle)) == 0
            if not ok:
                raise OSError("no NVML handle")
            self.lib, self.handle = lib, handle
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self._reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.nvml = True
        except Exception:
            self.nvml = False
        self.torch_index = torch_index

    def _run(self):
        # back-to-back queries with a short sleep between them; each sample carries
        # its host time so that the ones inside the timed window can be picked out
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self.lib.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(clk)) == 0 and \
                    self._reasons_fn(self.handle, ctypes.byref(rs)) == 0:
                self.samples.append((time.perf_counter(), clk.value, int(rs.value)))
            time.sleep(0.00005)

    def start(self):
        """Start sampling; returns once the first sample is in (so that a timed region
        that follows is covered from its start)."""
        if self.nvml:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()
            t0 = time.perf_counter()
            while not self.samples and time.perf_counter() - t0 < 2.0:
                time.sleep(0.0005)
        else:
            try:
                self._proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.torch_index),
                     "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                     "--format=csv,noheader,nounits", "-lms", "100"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except Exception:
                self._proc = None

    def stop(self, t_begin=None, t_end=None):
        """Stop sampling and summarise the samples taken between t_begin and t_end
        (host perf_counter times; all samples when not given)."""
        if self._thread:
            self._stop.set()
            self._thread.join()
        if self._proc:
            self._proc.terminate()
            out, _ = self._proc.communicate(timeout=5)
            now = time.perf_counter()
            for line in out.splitlines():
                try:
                    a, b, c = [x.strip() for x in line.split(",")]
                    self.max_mhz = float(b)
                    self.samples.append((now, float(a), int(c, 16)))
                except Exception:
                    pass
        sel = [x for x in self.samples
               if (t_begin is None or x[0] >= t_begin) and (t_end is None or x[0] <= t_end)]
        src = "nvml" if self.nvml else "nvidia-smi"
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "source": src}
        mask = 0
        for _, _, r in sel:
            mask |= r
        reasons = [n for bit, n in self.REASONS.items() if mask & bit and n != "gpu_idle"]
        return {"sm_mhz": statistics.median(c for _, c, _ in sel),
                "sm_min_mhz": min(c for _, c, _ in sel),
                "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(sel),
                "source": src}


def input_scales(x):
    """The dequantisation scales of an e4m3 workload's inputs (none for 16-bit ones)."""
    return {k: x[k] for k in ("q_scale", "kv_scale") if k in x}


def max_over_ranks(x, world, device):
    """The largest of every rank's `x` (the job's time is its slowest rank's)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world, flops_per_rank, ms):
    """Whole-job throughput: every rank's flops over the slowest rank's step time."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def oracle_sample_time(w, target_seconds, seqs_max=64):
    """Time the fp64 oracle (as it stands) on a bounded sample of workload `w`:
    whole sequences (all heads), drawn on the host, until ~target_seconds pass."""
    import numpy as np
    import oracle
    import workloads
    cores = os.cpu_count() or 1
    lens = [int(x) for x in w.seqlens]
    flops = 0.0
    nseq = 0
    elapsed = 0.0
    k = 0
    while elapsed < target_seconds and nseq < min(seqs_max, w.batch):
        L = lens[k % len(lens)]
        k += 1
        sub = workloads.custom(1, w.heads, (L,), w.dtype, w.page_size, w.softmax_scale,
                               seqlen_q=w.seqlen_q, causal=w.causal,
                               seed=1000 + k, name="sample")
        x = workloads.make_inputs(sub, "cpu")
        q = workloads.to_bits(x["q"]).reshape(1, sub.rows, -1)
        kv = workloads.to_bits(x["kv_cache"][:, :, 0])
        t0 = time.perf_counter()
        oracle.decode(q, kv, x["block_table"].numpy(), x["cache_seqlens"].numpy(),
                      w.softmax_scale, w.dtype, threads=cores, seqlen_q=sub.seqlen_q,
                      is_causal=sub.causal, **input_scales(x))
        elapsed += time.perf_counter() - t0
        flops += sub.flops()
        nseq += 1
    del np
    return flops, elapsed, cores, nseq


# ------------------------------------------------------------------------------- arms

def workload_config(w, args, world):
    """The `config` object of both arms' lines: the workload and how it is fed, not how
    this library launches it (that goes under `launch`)."""
    kv_mb = w.total_tokens * 576 * w.elem_bytes / 1e6
    copies = max(1, args.copies)
    return {"workload": w.name, "batch": w.batch, "heads": w.heads, "seqlen_q": w.seqlen_q,
            "causal": w.causal, "seqlen": int(w.seqlens[0]), "page_block_size": w.page_size,
            "block_table": "seeded random permutation" if w.shuffle else "identity (pages in order)",
            "softmax_scale": w.softmax_scale, "input_dtype": w.dtype, "layout": args.layout,
            "l2": f"{copies} rotating input sets, KV {kv_mb:.0f} MB each "
                  + ("(> 129 MB L2)" if kv_mb > 129 else "(within the 129 MB L2)"),
            "parallelism": f"replicas x{world}"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import workloads
    w = workloads.get(args.config)
    if args.batch is not None:
        w = workloads.get(args.config, batch=args.batch, seqlens=tuple(w.seqlens[:1]) * args.batch)
    cores = os.cpu_count() or 1
    # one step = the oracle on one whole sequence (all heads) of the workload; the
    # sequence is trimmed if needed so that warmup+steps stay within ~2 minutes.
    import oracle
    L0 = int(w.seqlens[0])

    def one(L, seed):
        sub = workloads.custom(1, w.heads, (L,), w.dtype, w.page_size, w.softmax_scale,
                               seqlen_q=w.seqlen_q, causal=w.causal,
                               seed=seed, name="ref")
        x = workloads.make_inputs(sub, "cpu")
        q = workloads.to_bits(x["q"]).reshape(1, sub.rows, -1)
        kv = workloads.to_bits(x["kv_cache"][:, :, 0])
        t0 = time.perf_counter()
        oracle.decode(q, kv, x["block_table"].numpy(), x["cache_seqlens"].numpy(),
                      w.softmax_scale, w.dtype, threads=cores, seqlen_q=sub.seqlen_q,
                      is_causal=sub.causal, **input_scales(x))
        return time.perf_counter() - t0, sub.flops()

    t_probe, _ = one(min(L0, 512), 1)
    per_tok = t_probe / min(L0, 512)
    budget = 120.0 / max(1, args.steps + args.warmup)
    L = max(64, min(L0, int(budget / max(per_tok, 1e-9))))
    for i in range(args.warmup):
        one(L, 10 + i)
    tot_t, tot_f = 0.0, 0.0
    for i in range(args.steps):
        t, f = one(L, 100 + i)
        tot_t += t
        tot_f += f
    value = tot_f / tot_t / 1e12
    sample = (f"per step: 1 sequence x {w.rows} query rows x {L} tokens of workload "
              f"'{w.name}' (fp64 C oracle, {cores} threads)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot_t / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, args, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch
    import torch.distributed as dist

    import mla_decode_gb300 as mla
    import workloads

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = workloads.get(args.config)
    if args.batch is not None:
        w = workloads.get(args.config, batch=args.batch, seqlens=tuple(w.seqlens[:1]) * args.batch)

    # ---- inputs: `copies` sets that differ in where their KV cache lives
    base = workloads.make_inputs(w, dev)
    sets = [base]
    for _ in range(max(0, args.copies - 1)):
        sets.append({"q": base["q"].clone(), "kv_cache": base["kv_cache"].clone(),
                     "block_table": base["block_table"], "cache_seqlens": base["cache_seqlens"],
                     **input_scales(base)})
    sets = [as_layout(s, args.layout) for s in sets]
    base = sets[0]
    num_sm = mla.mla_device_num_sm(local)
    parts, stride = mla.mla_metadata_shape(w.batch, w.rows, num_sm)
    meta = torch.empty((parts, stride), dtype=torch.int32, device=dev)
    nsplit = torch.empty((w.batch + 1,), dtype=torch.int32, device=dev)
    combine = args.combine
    if combine == "auto":
        # every input set shares the batch's lengths, so one schedule decides for all
        mla.prepare_metadata(base["cache_seqlens"], w.heads, num_sm, meta, nsplit,
                             seqlen_q=w.seqlen_q)()
        combine = "fused" if int(nsplit[-1]) == w.batch else "kernel"
    ws = torch.empty((mla.mla_workspace_size(w.batch, w.rows, parts),), dtype=torch.uint8,
                     device=dev)
    out = torch.empty((w.batch, w.seqlen_q, w.heads, 512), dtype=mla.out_dtype(w.torch_dtype),
                      device=dev)
    lse = torch.empty((w.batch, w.heads) if w.seqlen_q == 1 else (w.batch, w.seqlen_q, w.heads),
                      dtype=torch.float32, device=dev)
    calls = [mla.prepare_decode(s["q"], s["kv_cache"], s["block_table"], s["cache_seqlens"],
                                w.softmax_scale, meta, nsplit, out, lse, ws, q_pe=s["q_pe"],
                                k_pe=s["k_pe"], is_causal=w.causal, **input_scales(s),
                                fused_combine=combine == "fused")
             for s in sets]
    metas = [mla.prepare_metadata(s["cache_seqlens"], w.heads, num_sm, meta, nsplit,
                                  seqlen_q=w.seqlen_q) for s in sets]

    def step(i, events=None):
        metas[i % len(metas)]()
        calls[i % len(calls)](split_events=events)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    code, detail = mla.mla_get_device_error()
    if code != 0:
        raise RuntimeError(f"device error {code} detail {detail}")

    K = args.steps
    # the split kernel's duration: CUDA events recorded around it on a sample of the
    # timed steps, one in the middle of every EVENT_EVERY (steps 5, 15, ...; step 0 when
    # K <= 5).  An event between two kernels ends the programmatic overlap of the second
    # one's launch with the first one's tail, so events on every step would add their
    # cost to every step
    timed = [i for i in range(K) if i % EVENT_EVERY == EVENT_EVERY // 2] or [0]
    ev = {i: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for i in timed}
    for a, b in ev.values():  # materialise the raw events
        a.record()
        b.record()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    h0 = time.perf_counter()
    # a fixed device-side delay ahead of the start event (outside the timed region), so
    # that the first steps are already queued when the GPU reaches it: the region then
    # holds the GPU work of the K steps, not the host's launch latency at its start
    torch.cuda._sleep(PREQUEUE_CYCLES)
    t0.record()
    for i in range(K):
        step(i, ev.get(i))
    t1.record()
    torch.cuda.synchronize()
    h1 = time.perf_counter()
    clk = clocks.stop(h0, h1)
    if world > 1:
        dist.barrier()
    ms = t0.elapsed_time(t1) / K
    split_ms = sum(a.elapsed_time(b) for a, b in ev.values()) / len(ev)
    code, detail = mla.mla_get_device_error()
    if code != 0:
        raise RuntimeError(f"device error {code} detail {detail}")
    ms = max_over_ranks(ms, world, dev)
    split_ms = max_over_ranks(split_ms, world, dev)

    # ---- end to end through the public API with pinned host buffers
    host = {k: v.cpu().pin_memory() for k, v in base.items() if torch.is_tensor(v)}
    dbuf = {k: torch.empty_like(base[k]) for k in host}
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    hlse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    e2e_call = mla.prepare_decode(dbuf["q"], dbuf["kv_cache"], dbuf["block_table"],
                                  dbuf["cache_seqlens"], w.softmax_scale, meta, nsplit, out, lse,
                                  ws, q_pe=dbuf.get("q_pe"), k_pe=dbuf.get("k_pe"),
                                  is_causal=w.causal, **input_scales(base),
                                  fused_combine=combine == "fused")
    e2e_meta = mla.prepare_metadata(dbuf["cache_seqlens"], w.heads, num_sm, meta, nsplit,
                                    seqlen_q=w.seqlen_q)
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = hout.numel() * hout.element_size() + hlse.numel() * hlse.element_size()

    def e2e_step():
        for k in dbuf:
            dbuf[k].copy_(host[k], non_blocking=True)
        e2e_meta()
        e2e_call()
        hout.copy_(out, non_blocking=True)
        hlse.copy_(lse, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    E = max(1, args.e2e_steps)
    if world > 1:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(E):
        e2e_step()
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / E
    e2e_ms = max_over_ranks(e2e_ms, world, dev)

    flops = w.flops()
    nbytes = w.bytes()
    hbm_peak, bf16_peak, peak_src = measured_peaks()
    achieved = nbytes / (split_ms * 1e-3) / 1e9
    traffic = ncu_traffic(w.name)
    # the bound is whichever of HBM bytes and tensor flops takes longer at the measured
    # peaks (fp16 runs at bf16's nominal tensor rate, e4m3 at twice it: 4.5 vs 2.25
    # PFLOP/s nominal); the kernel is timed alone in a ~100 us launch, so the burst
    # tensor peak applies
    f8 = w.dtype == "e4m3"
    tensor_peak = bf16_peak * (2.0 if f8 else 1.0)
    tflops_achieved = flops / (split_ms * 1e-3) / 1e12
    roofline = {"kernel": "split", "kernel_ms": split_ms, "kernel_launches_timed": len(ev),
                "traffic": traffic,
                "hbm_frac": achieved / hbm_peak, "tensor_frac": tflops_achieved / tensor_peak}
    if flops / (tensor_peak * 1e12) > nbytes / (hbm_peak * 1e9):
        roofline.update(bound="tensor", achieved=tflops_achieved, peak=tensor_peak, unit="TFLOP/s",
                        frac=tflops_achieved / tensor_peak,
                        peak_source=f"{peak_src} bf16_tflops (burst)"
                                    + (" x 2 (nominal e4m3 / bf16 ratio)" if f8 else ""))
    else:
        roofline.update(bound="hbm", achieved=achieved, peak=hbm_peak, unit="GB/s",
                        frac=achieved / hbm_peak, peak_source=f"{peak_src} hbm_gbs")
    line = {
        "metric": METRIC,
        "value": job_tflops(world, flops, ms),
        "unit": UNIT,
        "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic",
        "config": workload_config(w, args, world),
        "launch": {"num_sm_parts": parts, "combine": combine, "combine_choice": args.combine},
        "effective_hbm_gbs": world * nbytes / (ms * 1e-3) / 1e9,
        "roofline": roofline,
        "e2e": {"value": job_tflops(world, flops, e2e_ms), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": E,
                "ms_per_step": e2e_ms},
        # metadata, split and (unless fused) combine kernels per step
        "gpu_launches": (2 if combine == "fused" else 3) * K,
        "clocks": clk,
        "kernel_source_hash": kernel_source_hash(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        f, t, cores, nseq = oracle_sample_time(w, args.cpu_seconds)
        line["cpu_baseline"] = {
            "value": f / t / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{nseq} whole sequences x {w.rows} query rows of workload '{w.name}' "
                      f"(fp64 C oracle, {cores} threads, {t:.1f} s)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
