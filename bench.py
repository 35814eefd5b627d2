"""Benchmark: one decode step of paged attention on GB300 through the pa_v2 C ABI.

A step is the whole hot path for one batch: every sequence's newest token is written into the
cache and the decode attends over it -- by default one pa_v2_decode_append call (phase 1
writes the token while streaming its page, then the phase-2 combine); --decode two-kernel
runs pa_reshape_and_cache then pa_v2_decode, --decode fused pa_reshape_and_cache then
pa_v2_decode_fused (the combine by the last CTA of each (sequence, head group) inside phase
1).  The default workload is the largest decode batch,
MHA with ALiBi over a ragged batch (256 sequences, 16 heads, head size 96, block size 32,
lognormal lengths with median 1024 capped at 32768, bf16 query and cache: about 2.6 GB of
K and V per step); --workload picks another named workload.

Printed (rank 0, one JSON line): achieved HBM GB/s over the step (value), microseconds per
step, the phase-1 kernel's roofline fraction against the measured HBM copy bandwidth, an
end-to-end number through host buffers, SM clocks sampled during the timed region, and the
fp64 CPU oracle timed on a bounded sample of the same workload.

--impl reference times that oracle alone (the reference arm: there is no reference GPU
implementation of this path), on the host cores, for the same workload and metric.

Multi-GPU (torchrun): every rank runs its own independent batch (sequences shard across GPUs
with no data-path exchange); value = bytes of all ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode attn µs/step and achieved HBM GB/s (fraction of GB300 peak), 1 GPU"
DEFAULT_WORKLOAD = "mha_alibi_ragged"
L2_BYTES = 129 * 1024 * 1024
# each profiled kernel's sources: its committed ncu counters are valid while these are unchanged
_CSRC = os.path.join(ROOT, "paged_kv_cache_v2_gb300", "csrc")
KERNEL_SRCS = {
    "phase1": [os.path.join(_CSRC, f) for f in ("pa_phase1.cuh", "pa_kernels.cuh", "pa_ptx.cuh")],
    "prefix": [os.path.join(_CSRC, f) for f in ("pa_prefix.cuh", "pa_prefix_m256.cuh", "pa_prefix.h", "pa_tc.cuh",
                                                "pa_kernels.cuh", "pa_ptx.cuh")],
}
PROFILE_FILES = {"phase1": "pa_v2_phase1_{}.md", "prefix": "pa_prefix_{}.md"}
PROFILE_DIR = os.path.join(ROOT, "profiles")


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _kernel_hash(kernel: str = "phase1") -> str:
    h = hashlib.sha256()
    for path in KERNEL_SRCS[kernel]:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _profiled_traffic(workload: str, kernel: str = "phase1"):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(PROFILE_DIR, PROFILE_FILES[kernel].format(workload))
    try:
        txt = open(path).read()
    except OSError:
        return None
    h = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", txt)
    b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if not h or not b or h.group(1) != _kernel_hash(kernel):
        return None
    return float(b.group(1))


class _NvmlPoller:
    """SM clock and clock-event reasons read through NVML (read-only queries) every
    `period_s` from a thread, so that a timed region of a few milliseconds still gets samples.
    Reason bits: 0x4 sw_power_cap, 0x8 hw_slowdown, 0x20 sw_thermal_slowdown,
    0x40 hw_thermal_slowdown."""

    BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, torch_device_index: int, period_s: float = 0.0002):
        import ctypes

        self.period = period_s
        self.samples = []  # (sm_mhz, reasons bitmask)
        self.max_mhz = None
        self._stop = threading.Event()
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.lib = lib
        self.h = ctypes.c_void_p()
        ok = False
        try:
            import torch

            uuid = str(torch.cuda.get_device_properties(torch_device_index).uuid)
            name = (uuid if uuid.startswith("GPU-") else "GPU-" + uuid).encode()
            ok = lib.nvmlDeviceGetHandleByUUID(ctypes.c_char_p(name), ctypes.byref(self.h)) == 0
        except Exception:
            ok = False
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(torch_device_index), ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle")
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0:  # 1 = NVML_CLOCK_SM
            self.max_mhz = float(mx.value)
        fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self._reasons_fn = fn if fn is not None else lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self._ctypes = ctypes

    def _run(self):
        ct = self._ctypes
        mhz, rs = ct.c_uint(), ct.c_ulonglong()
        while not self._stop.is_set():
            if self.lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(mhz)) == 0:
                r = rs.value if self._reasons_fn(self.h, ct.byref(rs)) == 0 else 0
                self.samples.append((float(mhz.value), int(r)))
            time.sleep(self.period)

    def start(self):
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()

    def stop(self):
        self._stop.set()
        self._t.join(timeout=2)
        self.lib.nvmlShutdown()

    def summary(self):
        if not self.samples:
            return None
        sm = [s for s, _ in self.samples]
        reasons = sorted({n for _, r in self.samples for b, n in self.BITS.items() if r & b})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(sm), "sm_mhz_min": min(sm), "source": f"NVML every {self.period * 1e3:g} ms"}


class ClockSampler:
    """SM clock and throttle reasons sampled while the timed region runs: NVML polled every
    0.2 ms (the timed region of a short run lasts only milliseconds), and nvidia-smi at
    its 100 ms interval as a fallback when NVML cannot be loaded."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.nvml = None

    def __enter__(self):
        try:
            self.nvml = _NvmlPoller(self.gpu)
            self.nvml.start()
            return self
        except Exception:
            self.nvml = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def __exit__(self, *exc):
        if self.nvml is not None:
            self.nvml.stop()
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.nvml is not None:
            s = self.nvml.summary()
            if s is not None:
                return s
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "source": "nvidia-smi every 100 ms"}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def combine_ranks(step_bytes: float, ms_per_step: float, device, world: int):
    """Whole-job numbers of a multi-rank run: bytes summed over ranks, time of the slowest
    rank (each rank processes its own sequences; nothing else is exchanged)."""
    if world <= 1:
        return step_bytes, ms_per_step
    import torch
    import torch.distributed as dist

    t = torch.tensor([ms_per_step], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    b = torch.tensor([step_bytes], dtype=torch.float64, device=device)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(b.item()), float(t.item())


# decode e2e: steps a captured CUDA graph holds
GRAPH_STEPS = 4
SLEEP_CYCLES = 2_000_000  # about 1 ms of GPU time at the SM clock


def queue_ahead(stream=None):
    """Queue a GPU sleep ahead of a timed loop. With an empty queue the first timed step's
    events also measure the host submitting it (~0.2 ms against a ~0.09 ms decode step); with
    the device busy on the sleep, the host enqueues the first steps meanwhile and every timed
    step measures device time, as in a serving loop that keeps the queue fed. The sleep sits
    before the first event, outside every timed interval."""
    import torch
    with torch.cuda.stream(stream if stream is not None else torch.cuda.current_stream()):
        torch.cuda._sleep(SLEEP_CYCLES)


def _percentiles(xs, qs):
    """Nearest-rank percentiles of a list of floats."""
    ys = sorted(xs)
    return [ys[min(len(ys) - 1, max(0, int(round(q / 100 * (len(ys) - 1)))))] for q in qs]


def _oracle_tiny_1thread_us() -> float:
    """The oracle on the tiny decode workload (2 sequences of 37 and 600 tokens) on one host
    thread: median of five calls, in microseconds."""
    import oracle
    import workloads
    wl = workloads.make("tiny")
    ts = []
    for _ in range(5):
        t0 = time.perf_counter()
        oracle.decode_workload(wl, threads=1)
        ts.append(time.perf_counter() - t0)
    return round(sorted(ts)[2] * 1e6, 1)


def _cpu_baseline(wl, seconds: float, threads: int):
    """Time the fp64 oracle, sequence by sequence (all heads of each), cycling over the
    workload until about `seconds` of work is done; returns (GB/s, description, bytes, s)."""
    import numpy as np

    import oracle

    lens = wl.seq_lens.numpy()
    H = wl.num_heads
    per_tok = wl.num_kv_heads * wl.head_size * wl.kv_elem_bytes * 2
    qo = 2 * H * wl.head_size * wl.q_elem_bytes
    done_bytes, done_seqs, done_tok, t_total = 0, 0, 0, 0.0
    s = 0
    while t_total < seconds:
        pairs = np.array([(s, h) for h in range(H)], dtype=np.int32)
        t0 = time.perf_counter()
        oracle.decode_workload(wl, pairs=pairs, threads=threads)
        t_total += time.perf_counter() - t0
        done_bytes += int(lens[s]) * per_tok + qo
        done_tok += int(lens[s])
        done_seqs += 1
        s = (s + 1) % wl.num_seqs
    gbs = done_bytes / t_total / 1e9 if t_total > 0 else None
    desc = (f"oracle on {done_seqs} sequences of the workload in order, cycling ({done_seqs / wl.num_seqs:.2f} "
            f"passes; all {H} heads each, {done_tok} tokens), {t_total:.1f} s")
    return gbs, desc, done_bytes, t_total


def pack_inputs(tensors, device):
    """One pinned host buffer holding `tensors` (CPU) back to back at 256-byte offsets, a
    device buffer of the same size, and typed views of the device buffer shaped like them."""
    import torch

    offs, n = [], 0
    for t in tensors:
        offs.append(n)
        n += -(-t.numel() * t.element_size() // 256) * 256
    hbuf = torch.empty(n, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(n, dtype=torch.uint8, device=device)
    views = []
    for t, o in zip(tensors, offs):
        nb = t.numel() * t.element_size()
        hbuf[o:o + nb].copy_(t.contiguous().view(-1).view(torch.uint8))
        views.append(dbuf[o:o + nb].view(t.dtype).view(t.shape))
    return hbuf, dbuf, views


def workload_config(name: str, wl, world: int) -> dict:
    """The `config` object of a decode line: the workload's name and shape, the same for the
    GPU arm and the reference arm."""
    return {"workload": name, "num_seqs": wl.num_seqs, "num_heads": wl.num_heads,
            "num_kv_heads": wl.num_kv_heads, "head_size": wl.head_size, "block_size": wl.block_size,
            "kv_cache_dtype": wl.kv_cache_dtype, "tokens": int(wl.seq_lens.sum()), "max_seq_len": wl.max_seq_len,
            "bytes_per_step": int(wl.algorithmic_bytes() + wl.writer_bytes()),
            "parallelism": f"replicas x{world} (sequence shards)"}


def run_reference(args):
    """Reference arm: the CPU oracle, as it stands, on the host cores."""
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    import workloads

    threads = len(os.sched_getaffinity(0))
    wl = workloads.make(args.workload, canaries=False)
    per_step = []
    budget = max(0.5, 150.0 / max(1, args.steps + args.warmup))
    for i in range(args.warmup + args.steps):
        gbs, desc, nbytes, t = _cpu_baseline(wl, budget, threads)
        if i >= args.warmup:
            per_step.append((gbs, nbytes, t, desc))
    tot_b = sum(x[1] for x in per_step)
    tot_t = sum(x[2] for x in per_step)
    value = tot_b / tot_t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * tot_t / len(per_step), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.q_dtype if wl.kv_cache_dtype == "auto" else "fp8_e4m3",
        "data": "synthetic (seeded)",
        "config": workload_config(args.workload, wl, ws),
        "l2": "n/a (host)",
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": per_step[-1][3] + " per step"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch

    import paged_kv_cache_v2_gb300 as pa
    import workloads

    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    pa.load()

    wl = workloads.shard(args.workload, rank, ws, canaries=False) if ws > 1 else \
        workloads.make(args.workload, canaries=False)
    S, H, d = wl.query.shape
    # rotate between cache copies so that no step finds the previous steps' pages in L2: at
    # least two, and enough that the copies together span 2.5x the L2 (small batches)
    kv_bytes = wl.key_cache.numel() * wl.key_cache.element_size() * 2
    nrot = args.cache_copies or min(16, max(2, -(-int(2.5 * L2_BYTES) // kv_bytes)))
    kcs = [wl.key_cache.to(dev) for _ in range(nrot)]
    vcs = [wl.value_cache.to(dev) for _ in range(nrot)]
    q = wl.query.to(dev)
    bt, sl = wl.block_tables.to(dev), wl.seq_lens.to(dev)
    nk, nv, slots = wl.new_key.to(dev), wl.new_value.to(dev), wl.slot_mapping.to(dev)
    slopes = None if wl.alibi_slopes is None else wl.alibi_slopes.to(dev)
    out = torch.empty_like(q)
    tmp_dtype = q.dtype if args.tmp_dtype == "q" else torch.float32
    es, ml, tmp = pa.workspace(S, H, d, wl.max_seq_len, dev, tmp_dtype)
    # per-tensor scales, or (--head-scales) the same values as one scale per kv head, which
    # takes the per-head entry points
    ks, vs = wl.k_scale, wl.v_scale
    if args.head_scales:
        ks = torch.full((wl.num_kv_heads,), wl.k_scale, dtype=torch.float32, device=dev)
        vs = torch.full((wl.num_kv_heads,), wl.v_scale, dtype=torch.float32, device=dev)
    # the fused entry point's arrival counters: zeroed once, left at zero by every call
    ctr = pa.decode_counters(S, H, wl.num_kv_heads, dev) if args.decode == "fused" else None
    # scratch for the append entry's grid order (longest sequences first where CTAs stride);
    # filled with -1, so that after the warm-up it shows whether the library launched the
    # order kernel
    order = torch.full((S,), -1, dtype=torch.int32, device=dev) if args.order else None
    stream = torch.cuda.current_stream()

    def step(i, inp=None, out_=None):
        q_, bt_, sl_, nk_, nv_, slots_ = (q, bt, sl, nk, nv, slots) if inp is None else inp
        o_ = out if out_ is None else out_
        kc, vc = kcs[i % nrot], vcs[i % nrot]
        if args.decode == "append":
            # the writer of the newest token fused into the decode
            pa.pa_v2_decode_append(o_, es, ml, tmp, q_, nk_, nv_, kc, vc, wl.num_kv_heads, wl.scale, bt_, sl_,
                                   wl.block_size, wl.max_seq_len, slopes, wl.kv_cache_dtype, ks, vs,
                                   order=order)
            return
        pa.pa_reshape_and_cache(nk_, nv_, kc, vc, slots_, wl.kv_cache_dtype, ks, vs)
        pa.pa_v2_decode(o_, es, ml, tmp, q_, kc, vc, wl.num_kv_heads, wl.scale, bt_, sl_, wl.block_size,
                        wl.max_seq_len, slopes, wl.kv_cache_dtype, ks, vs, counters=ctr)

    decode_bytes = wl.algorithmic_bytes()
    step_bytes = decode_bytes + wl.writer_bytes()
    kv_q_bytes = decode_bytes - S * H * d * wl.q_elem_bytes  # phase-1 share: K, V and Q
    # writer + phase 1 (+ phase 2 on the two-kernel path; the fused path with an fp32
    # tmp_output always runs the combine inside phase 1)
    launches_per_step = (1 if args.decode == "append" else 2) + (1 if wl.max_num_partitions > 1 and ctr is None else 0)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    ordered = order is not None and args.decode == "append" and bool((order >= 0).all().item())
    launches_per_step += 1 if ordered else 0

    def barrier():
        if ws > 1:
            torch.distributed.barrier()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in kev:  # create the CUDA events (torch creates them lazily on first record)
        a.record(stream)
        b.record(stream)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clocks:
        # (a) the steps themselves, back to back, one event pair per step
        queue_ahead(stream)
        t_wall0 = time.perf_counter()
        for i in range(args.steps):
            ev[i][0].record(stream)
            step(args.warmup + i)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall0
        barrier()
        # (b) the same steps with events around the phase-1 launch (the library records them
        # on the launching stream); the extra events between kernels cost the launch overlap,
        # so (a) alone gives the step time.
        queue_ahead(stream)
        for i in range(args.steps):
            pa.pa_v2_set_timing_events(kev[i][0], kev[i][1])
            step(args.warmup + i)
        pa.pa_v2_set_timing_events(None, None)
        torch.cuda.synchronize()
    barrier()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    k_ms = [a.elapsed_time(b) for a, b in kev]
    # The event clock ticks in about 2 us here, so the mean step comes from the span of all K
    # back-to-back steps (first start to last end); the per-step times give the spread only.
    mean_ms = ev[0][0].elapsed_time(ev[-1][1]) / len(ev)
    all_bytes, mean_ms_max = combine_ranks(float(step_bytes), mean_ms, dev, ws)
    value = all_bytes / (mean_ms_max * 1e-3) / 1e9

    # ---- end to end through host buffers (pinned), same metric --------------------------
    e2e = None
    if not args.no_e2e:
        # The step's inputs travel in one pinned host buffer and one copy (a serving loop
        # stages them together), the output back in one copy.
        srcs = [wl.query, wl.block_tables, wl.seq_lens, wl.new_key, wl.new_value]
        if args.decode != "append":  # the append step takes the slots from the tables
            srcs.append(wl.slot_mapping)
        tail = () if args.decode != "append" else (slots,)
        hbuf, dbuf, views = pack_inputs(srcs, dev)
        dbuf2 = torch.empty_like(dbuf)
        views2 = [dbuf2[v.data_ptr() - dbuf.data_ptr():][:v.numel() * v.element_size()].view(v.dtype).view(v.shape)
                  for v in views]
        inps = (tuple(views) + tail, tuple(views2) + tail)
        outs = (out, torch.empty_like(out))
        houts = tuple(torch.empty_like(wl.query).pin_memory() for _ in range(2))
        h2d = sum(t.numel() * t.element_size() for t in srcs)
        d2h = houts[0].numel() * houts[0].element_size()
        dbufs = (dbuf, dbuf2)

        def e2e_serial(i):
            dbuf.copy_(hbuf, non_blocking=True)
            step(i, inps[0], outs[0])
            houts[0].copy_(outs[0], non_blocking=True)

        # Pipelined: a second stream carries step i+1's inputs in and step i's output out
        # while step i runs, with two device input buffers and two outputs (ping-pong).
        # Every step still copies its own inputs from pinned host memory and reads its
        # own output back inside the timed region.
        cstream = torch.cuda.Stream(dev)
        h2d_done = [torch.cuda.Event() for _ in range(2)]
        step_done = [torch.cuda.Event() for _ in range(2)]
        d2h_done = [torch.cuda.Event() for _ in range(2)]

        def e2e_pipelined(i0, n):
            cur = torch.cuda.current_stream()  # the compute stream (a capture stream in a graph)
            cstream.wait_stream(cur)
            with torch.cuda.stream(cstream):
                dbufs[0].copy_(hbuf, non_blocking=True)
                h2d_done[0].record(cstream)
            for j in range(n):
                b = j % 2
                cur.wait_event(h2d_done[b])
                if j >= 2:  # the output buffer's previous read-back has finished
                    cur.wait_event(d2h_done[b])
                step(i0 + j, inps[b], outs[b])
                step_done[b].record(cur)
                with torch.cuda.stream(cstream):
                    if j + 1 < n:  # the other input buffer was last read by step j-1,
                        # whose read-back below already waited for it on this stream
                        dbufs[1 - b].copy_(hbuf, non_blocking=True)
                        h2d_done[1 - b].record(cstream)
                    cstream.wait_event(step_done[b])
                    houts[b].copy_(outs[b], non_blocking=True)
                    d2h_done[b].record(cstream)
            cur.wait_stream(cstream)

        # Graphs: GRAPH_STEPS steps with their copies per graph, pipelined as above inside it;
        # one graph per stretch of the cache-copy rotation, each replayed in turn (one host
        # launch per GRAPH_STEPS steps).
        graphs, graph_error = [], None
        if args.graphs:
            try:
                for k in range(nrot // math.gcd(nrot, GRAPH_STEPS)):
                    e2e_pipelined(GRAPH_STEPS * k, GRAPH_STEPS)  # eager once: kernel attributes are set
                    torch.cuda.synchronize()
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g):
                        e2e_pipelined(GRAPH_STEPS * k, GRAPH_STEPS)
                    graphs.append(g)
                torch.cuda.synchronize()
            except RuntimeError as exc:  # reported in the line; the eager schedules stand
                graphs, graph_error = [], str(exc).splitlines()[0][:200]
        n_replays = -(-args.steps // GRAPH_STEPS)

        def replay_all():
            for j in range(n_replays):
                graphs[j % len(graphs)].replay()

        def timed(fn, nsteps=args.steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            barrier()
            torch.cuda.synchronize()
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            barrier()
            return combine_ranks(float(step_bytes), e0.elapsed_time(e1) / nsteps, dev, ws)[1]

        for i in range(max(1, args.warmup)):
            e2e_serial(i)
        e2e_pipelined(0, max(3, args.warmup))
        torch.cuda.synchronize()
        if graphs:
            replay_all()
        torch.cuda.synchronize()
        sched = {"serial": (timed(lambda: [e2e_serial(i) for i in range(args.steps)]),
                            "eager calls; the copies on the compute stream, before and after each step"),
                 "pipelined": (timed(lambda: e2e_pipelined(0, args.steps)),
                               "eager calls; a second stream, double-buffered: step i+1's inputs in and "
                               "step i's output out while step i runs")}
        if graphs:
            sched["graphs"] = (timed(replay_all, GRAPH_STEPS * n_replays),
                               f"CUDA graphs of {GRAPH_STEPS} steps each with their copies (pipelined "
                               "within the graph), replayed")
        best = min(sched, key=lambda k: sched[k][0])
        e_ms = sched[best][0]
        e2e = {"value": round(all_bytes / (e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
               "us_per_step": round(e_ms * 1e3, 2), "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "schedule": best,
               "schedules": {k: {"value": round(all_bytes / (v[0] * 1e-3) / 1e9, 2),
                                 "us_per_step": round(v[0] * 1e3, 2), "how": v[1]} for k, v in sched.items()}}
        if graph_error:
            e2e["graph_capture_failed"] = graph_error

    if rank != 0:
        if ws > 1:
            torch.distributed.destroy_process_group()
        return 0

    peak, peak_kind = _peaks()
    k_mean = sum(k_ms) / len(k_ms)
    achieved = kv_q_bytes / (k_mean * 1e-3) / 1e9
    traffic = _profiled_traffic(args.workload)
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "us_per_step": round(mean_ms_max * 1e3, 2),
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(mean_ms_max, 5),
        # this rank's per-step spread (CUDA events around each step)
        "us_p10_p50_p90": [round(float(x) * 1e3, 2) for x in _percentiles(step_ms, (10, 50, 90))],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": wl.q_dtype if wl.kv_cache_dtype == "auto" else f"{wl.q_dtype}+fp8_e4m3",
        "data": "synthetic (seeded N(0, sigma) values, random block tables)",
        "config": workload_config(args.workload, wl, ws),
        "scales": "one k_scale / v_scale per kv head (the head-scales entry points)" if args.head_scales
                  else "per tensor",
        "tmp_output": "query dtype" if args.tmp_dtype == "q" else "float32",
        "decode_entry": {"append": "pa_v2_decode_append", "fused": "pa_v2_decode_fused"}.get(args.decode,
                                                                                               "pa_v2_decode"),
        "grid_order": "longest-first (pa_v2_decode_order inside the call)" if ordered else "index order",
        "fraction_of_peak": round(value / peak, 4),
        "l2": f"{decode_bytes / 2**20:.0f} MiB of K/V read per step from {nrot} rotating cache copies of "
              f"{kv_bytes / 2**20:.0f} MiB ({nrot * kv_bytes / L2_BYTES:.1f}x the L2 together)",
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": "pa_v2_phase1_kernel", "kernel_us": round(k_mean * 1e3, 2),
                     "bytes_per_launch": int(kv_q_bytes), "peak_source": f"{peak_kind} hbm_gbs (copy)"},
        "cpu_baseline": None,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks.summary(),
        "wall_s_timed_region": round(t_wall, 4),
    }
    if ws == 1 and not args.no_cpu_baseline:
        threads = len(os.sched_getaffinity(0))
        gbs, desc, _, _ = _cpu_baseline(wl, args.cpu_seconds, threads)
        line["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                                "sample": desc, "tiny_1thread_us": _oracle_tiny_1thread_us()}
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_copy_blocks(args):
    """Copy-on-write block copies ("paged_attn.py" copy_blocks): 32 layers of fp16 K/V caches
    (8 kv heads x head size 128 x block size 16 = 32 KiB per block and cache), 512 random
    (src, dst) pairs per step; bytes = read + write of every copied block."""
    import torch

    import paged_kv_cache_v2_gb300 as pa

    torch.cuda.set_device(0)
    pa.load()
    L, NB, pairs = 32, 2048, 512
    g = torch.Generator(device="cuda").manual_seed(11)
    kcs = [torch.empty((NB, 8, 16, 16, 8), dtype=torch.float16, device="cuda").normal_(generator=g) for _ in range(L)]
    vcs = [torch.empty((NB, 8, 128, 16), dtype=torch.float16, device="cuda").normal_(generator=g) for _ in range(L)]
    perm = torch.randperm(NB, device="cuda", generator=g)
    maps = [torch.stack([perm[:pairs], perm[pairs:2 * pairs]], 1).contiguous(),
            torch.stack([perm[2 * pairs:3 * pairs], perm[3 * pairs:]], 1).contiguous()]
    block = kcs[0][0].numel() * 2
    step_bytes = L * pairs * 2 * block * 2
    for i in range(args.warmup):
        pa.pa_copy_blocks(kcs, vcs, maps[i % 2])
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(0) as clocks:
        queue_ahead()
        for i in range(args.steps):
            ev[i][0].record()
            pa.pa_copy_blocks(kcs, vcs, maps[i % 2])
            ev[i][1].record()
        torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    peak, kind = _peaks()
    gbs = step_bytes / (ms * 1e-3) / 1e9
    print(json.dumps({
        "metric": "copy_blocks achieved HBM GB/s (read + write of copied blocks), 1 GPU", "value": round(gbs, 1),
        "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": "copy_blocks 32 layers x 512 pairs x 32 KiB blocks (K and V)",
                   "bytes_per_step": step_bytes, "l2": f"{step_bytes / 2**20:.0f} MiB per step, > L2"},
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(gbs / peak, 4), "traffic": None, "kernel": "pa_copy_blocks_kernel",
                     "peak_source": f"{kind} hbm_gbs (copy)"},
        "gpu_launches": args.steps, "clocks": clocks.summary()}), flush=True)
    return 0


def run_swap_blocks(args):
    """Block swaps between the GPU cache and a pinned host cache ("paged_attn.py" swap_blocks):
    fp16 blocks of 32 KiB (8 kv heads x head size 128 x block size 16), 512 random blocks out
    (GPU -> host) and 512 in (host -> GPU) per step; bytes = every moved block once.  The
    roofline's peak is the same bytes moved as one contiguous copy each way, timed in the same
    run (the host link's rate for large copies)."""
    import torch

    import paged_kv_cache_v2_gb300 as pa

    torch.cuda.set_device(0)
    pa.load()
    NB, pairs = 4096, 512
    g = torch.Generator().manual_seed(12)
    gpu = torch.empty((NB, 8, 128, 16), dtype=torch.float16, device="cuda").normal_()
    host = torch.empty((NB, 8, 128, 16), dtype=torch.float16).pin_memory()
    host.normal_()
    block = gpu[0].numel() * 2
    step_bytes = 2 * pairs * block
    perms = [torch.randperm(NB, generator=g) for _ in range(2)]
    outs = [torch.stack([p[:pairs], p[pairs:2 * pairs]], 1).contiguous() for p in perms]
    ins = [torch.stack([p[2 * pairs:3 * pairs], p[3 * pairs:4 * pairs]], 1).contiguous() for p in perms]

    def step(i):
        pa.pa_swap_blocks(gpu, host, outs[i % 2])
        pa.pa_swap_blocks(host, gpu, ins[i % 2])

    dbig = torch.empty(pairs * block, dtype=torch.uint8, device="cuda")
    hbig = torch.empty(pairs * block, dtype=torch.uint8).pin_memory()

    def contiguous():
        hbig.copy_(dbig, non_blocking=True)
        dbig.copy_(hbig, non_blocking=True)

    def timed(fn):
        for i in range(args.warmup):
            fn(i)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        a.record()
        for i in range(args.steps):
            fn(i)
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / args.steps, (time.perf_counter() - t0) * 1e3 / args.steps

    with ClockSampler(0) as clocks:
        ms, host_ms = timed(step)
        ref_ms, _ = timed(lambda i: contiguous())
    gbs = step_bytes / (ms * 1e-3) / 1e9
    ref = step_bytes / (ref_ms * 1e-3) / 1e9
    print(json.dumps({
        "metric": "swap_blocks achieved host-link GB/s (blocks out + blocks in), 1 GPU", "value": round(gbs, 1),
        "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "host_ms_per_step": round(host_ms, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16", "data": "synthetic",
        "config": {"workload": "swap_blocks 512 blocks out + 512 in, 32 KiB blocks, pinned host cache",
                   "bytes_per_step": step_bytes},
        "roofline": {"bound": "host link", "achieved": round(gbs, 1), "peak": round(ref, 1), "unit": "GB/s",
                     "frac": round(gbs / ref, 4), "traffic": None, "kernel": "pa_swap_blocks_kernel",
                     "peak_source": "one contiguous copy of the same bytes each way, this run"},
        # one launch per 480 pairs and direction (the library's kernel path for pinned memory)
        "gpu_launches": 2 * -(-pairs // 480) * args.steps, "clocks": clocks.summary()}), flush=True)
    return 0


def _tensor_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def run_prefix(args):
    """Chunked-prefix attention ("paged_attn.py" forward_prefix) on one chunked-prefill step:
    every new token attends to its sequence's cached context and causally to its chunk.
    value = algorithmic TFLOP/s (4 d H per visible (query, key) pair) of the pa_prefix call;
    roofline against the measured dense bf16 tensor throughput (fp16 runs at the same rate)."""
    import numpy as np
    import torch

    import paged_kv_cache_v2_gb300 as pa
    import workloads

    name = args.workload if args.workload in workloads.PREFIX_CONFIGS else "prefix_long_gqa"
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev_i = torch.cuda.current_device()
    pa.load()
    # each rank runs its own step of the same shape (sequences are independent: weak scaling)
    wl = workloads.make_prefix(name, seed=workloads.PREFIX_CONFIGS[name]["seed"] + 100_003 * rank) if ws > 1 \
        else workloads.make_prefix(name)
    dev = {k: getattr(wl, k).cuda() for k in ("query", "key", "value", "key_cache", "value_cache",
                                              "block_tables", "query_start_loc", "context_lens")}
    out = torch.empty_like(dev["query"])
    flops = wl.flops()
    # contexts longer than 16384 tokens are cut into up to 8 parts (the binding's defaults;
    # --min-split-keys / --max-splits change them);
    # the workspace for their partial results is allocated once, outside the timed region
    split_keys = args.min_split_keys or pa.PREFIX_SPLIT_KEYS
    max_splits = max(1, min(args.max_splits, -(-wl.block_tables.shape[1] * wl.block_size // split_keys)))
    ws_bytes = pa.prefix_workspace_size(wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_size,
                                        wl.max_query_len, max_splits)
    work = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda") if ws_bytes else None

    def call(q, k, v, o):
        pa.pa_prefix(o, q, k, v, dev["key_cache"], dev["value_cache"], dev["block_tables"],
                     dev["query_start_loc"], dev["context_lens"], wl.max_query_len, scale=wl.scale,
                     workspace=work, max_splits=max_splits, min_split_keys=args.min_split_keys)

    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
    for _ in range(args.warmup):
        call(dev["query"], dev["key"], dev["value"], out)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
        torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in kev:  # create the CUDA events (torch creates them lazily on first record)
        a.record()
        b.record()
    torch.cuda.synchronize()
    parts = pa.prefix_num_parts(wl.num_heads, wl.num_kv_heads, wl.head_size, dev["query"].dtype, wl.max_query_len,
                                wl.block_tables.shape[1], wl.block_size, max_splits, args.min_split_keys,
                                work is not None)
    n_kernels = 2 if parts > 1 else 1  # the attention kernel (+ the combine of split contexts)
    launches = 0
    with ClockSampler(dev_i) as clocks:
        queue_ahead()
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record()
            pa.pa_v2_set_timing_events(kev[i][0], kev[i][1])  # the library records them around the attention kernel
            call(dev["query"], dev["key"], dev["value"], out)
            ev[i][1].record()
            launches += n_kernels
        pa.pa_v2_set_timing_events(None, None)
        torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    times = sorted(a.elapsed_time(b) for a, b in ev)
    ms_rank = sum(times) / len(times)
    k_ms = sum(a.elapsed_time(b) for a, b in kev) / args.steps
    all_flops, ms = combine_ranks(float(flops), ms_rank, torch.device("cuda", dev_i), ws)
    tflops = all_flops / (ms * 1e-3) / 1e12
    rank_tflops = flops / (k_ms * 1e-3) / 1e12
    e2e = None
    if not args.no_e2e:
        # the step's q/k/v rows in one pinned host buffer and one copy, the output back in one
        srcs = [getattr(wl, k) for k in ("query", "key", "value")]
        hbuf, dbuf, (dq, dk, dv) = pack_inputs(srcs, dev["query"].device)
        ho = torch.empty(wl.query.shape, dtype=wl.query.dtype).pin_memory()
        for _ in range(2):
            dbuf.copy_(hbuf, non_blocking=True)
            call(dq, dk, dv, out)
            ho.copy_(out, non_blocking=True)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.steps):
            dbuf.copy_(hbuf, non_blocking=True)
            call(dq, dk, dv, out)
            ho.copy_(out, non_blocking=True)
            launches += n_kernels
        b.record()
        torch.cuda.synchronize()
        e_ms = a.elapsed_time(b) / args.steps
        if ws > 1:
            _, e_ms = combine_ranks(0.0, e_ms, torch.device("cuda", dev_i), ws)
        h2d = sum(t.numel() * t.element_size() for t in srcs)
        e2e = {"value": round(all_flops / (e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms_per_step": round(e_ms, 4),
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": ho.numel() * ho.element_size()}
    cpu = None
    if not args.no_cpu_baseline and rank == 0 and ws == 1:
        import oracle
        threads = len(os.sched_getaffinity(0))
        qsl = wl.query_start_loc.numpy()
        rng = np.random.default_rng(0)
        done_flops, t_total, nrows = 0, 0.0, 0
        while t_total < args.cpu_seconds:
            tok = int(rng.integers(0, wl.num_tokens))
            s = int(np.searchsorted(qsl, tok, side="right") - 1)
            rows = np.array([(tok, h) for h in range(wl.num_heads)], dtype=np.int32)
            t0 = time.perf_counter()
            oracle.prefix_workload(wl, rows=rows, threads=threads)
            t_total += time.perf_counter() - t0
            keys = int(wl.context_lens[s]) + tok - int(qsl[s]) + 1
            done_flops += 4 * wl.head_size * wl.num_heads * keys
            nrows += wl.num_heads
        cpu = {"value": round(done_flops / t_total / 1e12, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"fp64 oracle on {nrows} (token, head) rows: all heads of random new tokens of the "
                         f"workload, {t_total:.1f} s"}
    peak, kind = _tensor_peak()
    if rank != 0:
        if ws > 1:
            torch.distributed.destroy_process_group()
        return 0
    print(json.dumps({
        "metric": f"chunked-prefix attention TFLOP/s (4 d H per visible query-key pair), {ws} GPU",
        "value": round(tflops, 2), "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": wl.q_dtype, "data": "synthetic",
        "config": {"workload": name, "num_seqs": wl.num_seqs, "heads": [wl.num_heads, wl.num_kv_heads],
                   "head_size": wl.head_size, "block_size": wl.block_size,
                   "context_lens": wl.context_lens.tolist(), "query_lens": wl.query_lens.tolist(),
                   "flops_per_step": flops, "l2": "flushed (256 MiB write) before every timed call",
                   "max_splits": max_splits, "min_split_keys": split_keys, "context_parts": parts,
                   "parallelism": f"replicas x{ws} (sequence shards)"},
        "roofline": {"bound": "tensor", "achieved": round(rank_tflops, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(rank_tflops / peak, 4), "traffic": _profiled_traffic(name, "prefix"),
                     "kernel": "pa_prefix_m256_kernel" if wl.head_size <= 128 else "pa_prefix_kernel",
                     "kernel_ms": round(k_ms, 4),
                     "peak_source": f"{kind} bf16_tflops (burst; fp16 has the same dense rate)"},
        "e2e": e2e, "cpu_baseline": cpu, "gpu_launches": launches, "clocks": clocks.summary()}), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graphs", dest="graphs", action="store_false",
                    help="decode e2e: time the eager schedules only (no CUDA-graph capture of the step)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--decode", choices=["append", "fused", "two-kernel"], default="append",
                    help="decode entry point: pa_v2_decode_append (the newest token's cache write inside phase "
                         "1, the default), pa_v2_decode after pa_reshape_and_cache (two-kernel), or "
                         "pa_v2_decode_fused (the combine by the last CTA inside phase 1 on grids of at most "
                         "two waves; measured slower on every workload here)")
    ap.add_argument("--head-scales", action="store_true",
                    help="decode: pass the scales as one per kv head (the head-scales entry points)")
    ap.add_argument("--tmp-dtype", choices=["f32", "q"], default="f32",
                    help="decode: tmp_output in float32 (default) or in the query dtype")
    ap.add_argument("--no-order", dest="order", action="store_false",
                    help="decode (append): no grid-order scratch, so the grid serves sequences in index order")
    ap.add_argument("--cache-copies", type=int, default=0,
                    help="decode: copies of the K/V caches the steps rotate through (0: at least 2 and enough "
                         "to span 2.5x the L2, so no step finds earlier steps' pages there; 1 for profiler runs)")
    ap.add_argument("--max-splits", type=int, default=8,
                    help="prefix: most parts a long context is cut into (1: no split)")
    ap.add_argument("--min-split-keys", type=int, default=0,
                    help="prefix: shortest context (keys, a multiple of 64) that is cut (0: the library's 16384)")
    ap.add_argument("--op", choices=["decode", "copy_blocks", "swap_blocks", "prefix"], default="decode",
                    help="decode: the decode step (default); copy_blocks: the block-copy kernel alone; "
                         "swap_blocks: block moves between the GPU cache and a pinned host cache; "
                         "prefix: chunked-prefix attention (--workload prefix_long_gqa|prefix_llama_gqa)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.op == "swap_blocks":
        return run_swap_blocks(args)
    if args.op == "copy_blocks":
        return run_copy_blocks(args)
    if args.op == "prefix":
        return run_prefix(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
