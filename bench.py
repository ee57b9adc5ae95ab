"""Decode-attention benchmark: KV GB/s, rows/s and HBM-roofline fraction.

One step = one pass of the whole hot path over one batch: split plan, split
kernel, combine (three launches through the C ABI), inputs resident in HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload long_context|gqa_paged|mla_sparse|tiny|...]

Prints one JSON line (rank 0).  Under torchrun each rank runs its own replica
of the workload (rows are independent; no collective on the data path) and
the step time is the max over ranks.  ``--impl reference`` times the fp64 CPU
oracle on the host cores on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import sys
import threading
import time

# numpy's BLAS threads for the CPU oracle leg: all host cores, stated in the output
_CORES = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(_CORES))

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

L2_FLUSH_BELOW = 256 << 20  # bytes; GB300 L2 is ~126 MB
METRIC = "decode-attn KV GB/s (% of GB300 HBM peak), rows/s; invariant vs balanced split"
PROFILE_DIR = os.path.join(ROOT, "profiles")
KERNEL_SOURCES = {
    "split_fma": ["invariant_decode_attention_gb300/csrc/split_fma.cu",
                  "invariant_decode_attention_gb300/csrc/common.cuh"],
    "split_gqa_tc": ["invariant_decode_attention_gb300/csrc/split_gqa_tc.cu",
                     "invariant_decode_attention_gb300/csrc/tcgen05.cuh",
                     "invariant_decode_attention_gb300/csrc/common.cuh"],
    "split_mla": ["invariant_decode_attention_gb300/csrc/split_mla.cu",
                  "invariant_decode_attention_gb300/csrc/tcgen05.cuh",
                  "invariant_decode_attention_gb300/csrc/common.cuh"],
}


# ----------------------------------------------------------------- helpers

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def tensor_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"])
    return 1900.0


def source_hash(kernel):
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(PROFILE_DIR, "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    r = rec.get(f"{kernel}:{workload}")
    if not r or r.get("src_sha") != source_hash(kernel):
        return None
    return r.get("dram_bytes_per_launch")


class ClockSampler:
    """Samples SM clock and throttle reasons through NVML while running."""

    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
               0x4: "sw_power_cap", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index=0, period=0.005):
        self.period = period
        self.samples, self.reasons, self.max_mhz = [], set(), None
        self._stop = threading.Event()
        self._nvml = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() == 0:
                h = ctypes.c_void_p()
                if nv.nvmlDeviceGetHandleByIndex_v2(device_index, ctypes.byref(h)) == 0:
                    self._nvml, self._h = nv, h
                    mx = ctypes.c_uint()
                    if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                        self.max_mhz = mx.value
        except OSError:
            pass

    def _run(self):
        nv, h = self._nvml, self._h
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                self.samples.append(clk.value)
            if nv.nvmlDeviceGetCurrentClocksEventReasons(h, ctypes.byref(rs)) == 0:
                for bit, name in self.REASONS.items():
                    if rs.value & bit:
                        self.reasons.add(name)
            time.sleep(self.period)

    def __enter__(self):
        if self._nvml is not None:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *exc):
        if self._nvml is not None:
            self._stop.set()
            self._t.join()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                    "samples": 0}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples)}


def max_over_ranks(x, device="cpu"):
    """The largest value of x over all ranks (x itself when not distributed);
    a barrier follows so no rank runs ahead into the next phase."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.barrier()
    return float(t.item())


def replica_value(per_rank_units, world, ms_per_step):
    """Whole-job throughput: units all ranks processed per second of the
    slowest rank's step (weak scaling: every rank runs its own batch)."""
    return world * per_rank_units / (ms_per_step * 1e-3)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# ----------------------------------------------------------------- workloads

def build_workload(name, rank=0):
    from invariant_decode_attention_gb300 import workloads as W
    seed_shift = 100 * rank  # every rank its own replica batch (weak scaling)
    if name == "gqa_paged":
        return W.gqa_paged(seed=1001 + seed_shift)
    if name == "long_context":
        return W.long_context(seed=1004 + seed_shift)
    if name == "tiny":
        return W.tiny(seed=1000 + seed_shift)
    if name == "mla_sparse":
        return W.mla_sparse(seed=1002 + seed_shift)
    if name == "mla_sparse_fp8":
        return W.mla_sparse_fp8(seed=1002 + seed_shift)
    if name == "gqa_paged_fp8":
        return W.gqa_paged_fp8(seed=1001 + seed_shift)
    if name == "long_context_fp8":
        return W.long_context_fp8(seed=1004 + seed_shift)
    if name == "gqa16_paged":
        return W.gqa16_paged(seed=1007 + seed_shift)
    if name == "gqa16_paged_fp8":
        return W.gqa16_paged_fp8(seed=1007 + seed_shift)
    if name == "gqa16_paged_nvfp4":
        return W.gqa16_paged_nvfp4(seed=1007 + seed_shift)
    if name == "gqa_paged_nvfp4":
        return W.gqa_paged_nvfp4(seed=1001 + seed_shift)
    if name == "long_context_nvfp4":
        return W.long_context_nvfp4(seed=1004 + seed_shift)
    raise ValueError(name)


class GpuCase:
    """A workload resident on the device plus its plan/run/combine step."""

    def __init__(self, wl_cpu, device, policy):
        from invariant_decode_attention_gb300 import api
        self.api = api
        self.cpu = wl_cpu
        self.wl = wl_cpu.to(device)
        self.policy = policy
        self.prob = api.problem_for(self.wl)
        self.ws = api.workspace(self.prob, device)
        self.out = torch.empty((self.wl.B, self.wl.H_q, self.wl.D_v), dtype=torch.bfloat16,
                               device=device)
        self.lse = torch.empty((self.wl.B, self.wl.H_q), dtype=torch.float32, device=device)

    def step(self, ev_run=None):
        a, w = self.api, self.wl
        pl = a.plan(self.prob, self.policy, w.lengths, self.ws)
        if ev_run is not None:
            ev_run[0].record()
        a.run(pl, w.q, w.k, w.v, w.table, w.lengths, self.out, self.lse)
        if ev_run is not None:
            ev_run[1].record()
        a.combine(pl, self.out, self.lse)


_FLUSH = None


def flush_l2():
    """Write a buffer twice the size of L2 so the next step starts cold."""
    global _FLUSH
    if _FLUSH is None:
        _FLUSH = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    _FLUSH.fill_(1)


def time_steps(case, steps, warmup, split_events=True, flush=False):
    """Device time per step (ms) and of the split kernel alone, CUDA events on
    the launching stream, synchronised on both sides.  With flush=True, L2 is
    flushed between steps (outside the events) and the total is the sum of
    the per-step event times."""
    for _ in range(warmup):
        case.step()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    runs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(steps)] if split_events else [None] * steps
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record()
    for i in range(steps):
        if flush:
            flush_l2()
        starts[i].record()
        case.step(runs[i])
        ends[i].record()
    t1.record()
    torch.cuda.synchronize()
    per_step = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    split = [r[0].elapsed_time(r[1]) for r in runs] if split_events else []
    total = sum(per_step) if flush else t0.elapsed_time(t1)
    return total, per_step, split


def packed_views(buf, specs):
    """Views of one contiguous byte buffer: specs is a list of (shape, dtype);
    each piece starts on a 256-byte boundary.  Returns the views in order."""
    views, off = [], 0
    for shape, dtype in specs:
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        views.append(buf[off:off + n].view(dtype).view(shape))
        off += (n + 255) // 256 * 256
    return views


def packed_bytes(specs):
    """Size of the buffer packed_views lays `specs` out in."""
    return sum((int(np.prod(s)) * torch.empty((), dtype=d).element_size() + 255) // 256 * 256
               for s, d in specs)


def e2e_steps(case, steps, warmup):
    """Same step through the public C entry point with host buffers: per step
    the step inputs (q, lengths, page table) go host->device from pinned
    memory and (out, lse) come back; the KV cache stays resident.  As a
    caller would, the inputs are staged in one pinned buffer and the outputs
    written into one device buffer, so each direction is one copy."""
    api, w = case.api, case.wl
    ins = [case.cpu.q, case.cpu.lengths] + ([] if case.cpu.table is None else [case.cpu.table])
    in_specs = [(tuple(t.shape), t.dtype) for t in ins]
    out_specs = [(tuple(case.out.shape), torch.bfloat16), (tuple(case.lse.shape), torch.float32)]
    h_in = torch.empty(packed_bytes(in_specs), dtype=torch.uint8).pin_memory()
    for v, t in zip(packed_views(h_in, in_specs), ins):
        v.copy_(t)
    d_in = torch.empty_like(h_in, device=case.out.device)
    d_views = packed_views(d_in, in_specs)
    d_q, d_len = d_views[0], d_views[1]
    d_tab = d_views[2] if len(d_views) > 2 else None
    d_outbuf = torch.empty(packed_bytes(out_specs), dtype=torch.uint8, device=case.out.device)
    d_out, d_lse = packed_views(d_outbuf, out_specs)
    h_outbuf = torch.empty(d_outbuf.numel(), dtype=torch.uint8).pin_memory()
    h2d, d2h = h_in.numel(), h_outbuf.numel()

    def one():
        d_in.copy_(h_in, non_blocking=True)
        api.forward(case.prob, case.policy, d_q, w.k, w.v, d_tab, d_len, case.ws, d_out, d_lse)
        h_outbuf.copy_(d_outbuf, non_blocking=True)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        one()
    b.record()
    torch.cuda.synchronize()
    # the staged result is the device step's result, bit for bit
    h_out, h_lse = packed_views(h_outbuf, out_specs)
    case.step()
    torch.cuda.synchronize()
    same = torch.equal(h_out, case.out.cpu()) and torch.equal(h_lse, case.lse.cpu())
    return a.elapsed_time(b) / steps, h2d, d2h, same


# ----------------------------------------------------------------- NVFP4 weight matmul

def nvfp4_section(api, peak, sizes=(1, 32, 33, 256), reps=30):
    """The NVFP4 weight matmul on the 8192 x 4096 projection: per row count n,
    the median device time of one call (rounding kernel + matmul kernel,
    captured once in a CUDA graph and replayed after an L2 flush), the
    weight-stream rate against the HBM copy peak and the matmul rate against
    the bf16 tensor peak; and whether one row's bits are the same at every n."""
    from invariant_decode_attention_gb300 import workloads as W
    codes, scales, gs = W.nvfp4_weight(8192, 4096, seed=1006)
    dc, ds = codes.cuda(), scales.cuda()
    wbytes = codes.numel() + scales.numel()
    pool = W.nvfp4_activations(max(sizes), 4096, seed=1006 + 7919).cuda()
    out, ref = {}, None
    for n in sizes:
        x = pool[:n].contiguous()
        ws = api.nvfp4_workspace(n, 8192, 4096)
        y = torch.empty((n, 8192), dtype=torch.float32, device="cuda")
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(3):
                api.nvfp4_mm(x, dc, ds, gs, y=y, ws=ws)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            api.nvfp4_mm(x, dc, ds, gs, y=y, ws=ws)
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        times = []
        for _ in range(reps):
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            graph.replay()
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        ms = statistics.median(times)
        flops = 2.0 * n * 8192 * 4096
        row = y[0].clone()
        ref = row if ref is None else ref
        out[f"n{n}"] = {
            "ms": round(ms, 5),
            "weight_gbs": round(wbytes / (ms * 1e-3) / 1e9, 1),
            "hbm_frac": round(wbytes / (ms * 1e-3) / 1e9 / peak, 4),
            "tflops": round(flops / (ms * 1e-3) / 1e12, 2),
            "tensor_frac_of_measured_bf16": round(flops / (ms * 1e-3) / 1e12 / tensor_peak(), 4),
            "row0_bits_equal_to_n1": bool(torch.equal(row, ref)),
        }
        del graph, ws, y
    return {"workload": "nvfp4_proj_N8192_K4096", "weight_bytes": wbytes,
            "timing": "CUDA graph of one call (rounding + matmul kernels), L2 flushed before "
                      "each replay, median of %d" % reps, "by_rows": out}


# ----------------------------------------------------------------- CPU oracle

def time_plan(case, steps):
    """Device time (ms) of the plan kernel alone: `steps` plan calls captured
    in one CUDA graph (so host-side call overhead is not timed), replayed
    between CUDA events."""
    a, w = case.api, case.wl
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            a.plan(case.prob, case.policy, w.lengths, case.ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(steps):
            a.plan(case.prob, case.policy, w.lengths, case.ws)
    graph.replay()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    graph.replay()
    e1.record()
    torch.cuda.synchronize()
    del graph
    return e0.elapsed_time(e1) / steps


def invariance_sweep(api, sizes=(1, 2, 4, 8, 16, 32, 64, 128, 256), steps=10):
    """The ragged sweep's target row (length 4096, GQA 32/8, d = 128) at a random
    position among log-uniform batchmates, against its solo run, under each
    policy: how many batches move any bit of its output or LSE, the largest
    output difference, the step time of every batch (the occupancy cost of
    the per-row split rule on ragged batches) and the plan kernel's own time."""
    from invariant_decode_attention_gb300 import workloads as W
    sweep = W.RaggedSweep(sizes)
    res = {"batch_sizes": list(sizes)}
    for name, pol in (("invariant", api.INVARIANT), ("balanced", api.BALANCED)):
        o_solo, l_solo = api.run_workload(sweep.solo(), policy=pol)
        moved, max_abs, ms, gbs, plan_ms = 0, 0.0, [], [], []
        for i in range(len(sizes)):
            wl, pos = sweep.batch(i)
            case = GpuCase(wl, wl.q.device, pol)  # already on the device: no copy
            tot, _, _ = time_steps(case, steps, 3, split_events=False)
            ms.append(round(tot / steps, 5))
            gbs.append(round(wl.kv_bytes() / (tot / steps * 1e-3) / 1e9, 1))
            plan_ms.append(round(time_plan(case, steps), 5))
            o, l = case.out, case.lse
            same = torch.equal(o[pos], o_solo[0]) and torch.equal(l[pos], l_solo[0])
            moved += 0 if same else 1
            max_abs = max(max_abs, (o[pos].float() - o_solo[0].float()).abs().max().item())
            del case
        res[name] = {"batches_moving_target_row": moved, "batches": len(sizes),
                     "max_absdiff_out": max_abs, "ms_per_step": ms, "kv_gbs": gbs,
                     "plan_ms": plan_ms}
    res["invariant_over_balanced_time"] = [
        round(a / b, 4) for a, b in zip(res["invariant"]["ms_per_step"],
                                        res["balanced"]["ms_per_step"])]
    del sweep
    torch.cuda.empty_cache()
    return res


def cpu_oracle_rate(wl, budget_s=15.0, max_rows=None, group=None, first_row=0, cycle=False):
    """Time the fp64 oracle, as it stands, on whole rows of the workload until
    the budget is spent (group=h: only the query heads of KV head h, a
    bounded sample of each row; cycle=True: start over at row 0 while budget
    is left).  Returns (GB/s, rows/s, rows done, seconds)."""
    from oracle import attention as A
    q = wl.q.double().numpy()
    table = None if wl.table is None else wl.table.numpy()

    class View:  # fp64 reads of the bf16 cache, row by row
        def __init__(self, t):
            self.t, self.shape = t, tuple(t.shape)

        def __getitem__(self, idx):
            idx = idx if isinstance(idx, tuple) else (idx,)
            idx = tuple(torch.as_tensor(np.asarray(i)) if not isinstance(i, (int, slice)) else i
                        for i in idx)
            return self.t[idx].double().numpy()

    K, V = View(wl.k), (None if wl.v is None else View(wl.v))
    n_kv = 1 if group is not None else wl.H_kv
    per_entry = n_kv * (wl.D_qk + (0 if wl.v is None else wl.D_v)) * 2
    G = wl.H_q // wl.H_kv
    heads = None if group is None else list(range(group * G, (group + 1) * G))
    done, nbytes = 0, 0
    t0 = time.perf_counter()
    n_rows = wl.B if max_rows is None else min(wl.B, max_rows)
    for i in range(10 ** 9 if cycle else n_rows):
        b = (first_row + i) % wl.B
        A.attend(q, K, V, wl.lengths.numpy(), scale=wl.scale, layout=wl.layout, table=table,
                 page_size=wl.page_size, d_v=wl.D_v, rows=[b], heads=heads)
        done += 1
        nbytes += int(wl.lengths[b]) * per_entry
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return nbytes / dt / 1e9, done / dt, done, dt


# ----------------------------------------------------------------- main

def cpu_model():
    """The host CPU's model name (x86: /proc/cpuinfo; Arm: lscpu), or the machine."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        import subprocess
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine()


def alg_bytes_of(wl):
    """Algorithmic bytes of one split-kernel launch: the rows' KV payload,
    q, and the final out (bf16) and lse (fp32)."""
    return wl.kv_bytes() + wl.q.numel() * 2 + wl.B * wl.H_q * (wl.D_v * 2 + 4)


def measure(case, peak, peak_kind, steps, warmup, world=1, dev="cpu", clocks=None):
    """Step time (INVARIANT, then BALANCED on the same inputs) and the split
    kernel's own time and roofline for one resident workload."""
    api, wl = case.api, case.wl
    kv_bytes = wl.kv_bytes()
    flush = kv_bytes < L2_FLUSH_BELOW  # inputs that fit in L2 are flushed out of it
    case.policy = api.INVARIANT
    if clocks is not None:
        with clocks:
            total_ms, _, _ = time_steps(case, steps, warmup, split_events=False, flush=flush)
    else:
        total_ms, _, _ = time_steps(case, steps, warmup, split_events=False, flush=flush)
    total_ms = max_over_ranks(total_ms, dev)
    ms = total_ms / steps
    # the split kernel alone: events on the launching stream around it
    _, _, split_ms = time_steps(case, max(20, steps // 2), 3, flush=flush)
    split_avg = max_over_ranks(sum(split_ms) / len(split_ms), dev)
    alg = alg_bytes_of(wl)
    kernel = ("split_mla" if wl.v is None else
              "split_gqa_tc" if api.split_constants(case.prob)[0] == api.VARIANT_GQA_TC else
              "split_fma")
    n_bal = max(20, steps // 4)
    case.policy = api.BALANCED
    bal_ms, _, _ = time_steps(case, n_bal, warmup, split_events=False, flush=flush)
    bal_ms = max_over_ranks(bal_ms, dev) / n_bal
    case.policy = api.INVARIANT
    rec = {
        "ms_per_step": round(ms, 5),
        "kv_gbs": round(replica_value(kv_bytes, world, ms) / 1e9, 2),
        "rows_per_s": round(world * wl.B / (ms * 1e-3), 1),
        "hbm_frac_step_of_" + peak_kind: round(kv_bytes / (ms * 1e-3) / 1e9 / peak, 4),
        "l2": (f"L2 flushed between steps ({kv_bytes / 1e6:.0f} MB of KV per step)" if flush
               else f"inputs larger than L2 ({kv_bytes / 1e6:.0f} MB of KV per step)"),
        "balanced": {"ms_per_step": round(bal_ms, 5),
                     "kv_gbs": round(kv_bytes / (bal_ms * 1e-3) / 1e9, 2),
                     "invariant_over_balanced_time": round(ms / bal_ms, 4)},
        "roofline": {
            "kernel": kernel, "bound": "hbm",
            "achieved": round(alg / (split_avg * 1e-3) / 1e9, 1),
            "peak": peak, "unit": "GB/s",
            "frac": round(alg / (split_avg * 1e-3) / 1e9 / peak, 4),
            "peak_kind": peak_kind,
            "traffic": recorded_traffic(kernel, wl.name),
            "alg_bytes_per_launch": alg,
            "split_ms_avg": round(split_avg, 5),
        },
    }
    if kernel in ("split_mla", "split_gqa_tc"):
        n_ent = int(wl.lengths.to(torch.int64).sum())
        if wl.extra_lengths is not None:
            n_ent += int(wl.extra_lengths.to(torch.int64).sum())
        flops = n_ent * wl.H_q * (wl.D_qk + wl.D_v) * 2
        tp = tensor_peak()
        rec["roofline_tensor"] = {
            "bound": "tensor", "achieved": round(flops / (split_avg * 1e-3) / 1e12, 1),
            "peak": tp, "unit": "TFLOP/s",
            "frac": round(flops / (split_avg * 1e-3) / 1e12 / tp, 4),
            "flops_per_launch": flops,
        }
    return rec


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long_context",
                    choices=["gqa_paged", "long_context", "tiny", "mla_sparse", "gqa_paged_fp8",
                             "long_context_fp8", "gqa_paged_nvfp4", "long_context_nvfp4",
                             "gqa16_paged", "gqa16_paged_fp8", "gqa16_paged_nvfp4",
                             "mla_sparse_fp8"])
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the secondary workloads and the CPU baseline")
    ap.add_argument("--nvfp4-only", type=int, nargs="+", metavar="ROWS",
                    help="time only the NVFP4 weight matmul at these row counts and print "
                         "its JSON")
    ap.add_argument("--nvfp4-reps", type=int, default=30)
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")
    if args.impl == "reference":
        return reference_arm(args, rank, world)

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from invariant_decode_attention_gb300 import api
    api.lib()
    peak, peak_kind = measured_peaks()
    if args.nvfp4_only:
        if rank == 0:
            print(json.dumps(nvfp4_section(api, peak, sizes=tuple(args.nvfp4_only),
                                           reps=args.nvfp4_reps)), flush=True)
        return

    wl = build_workload(args.workload, rank)
    case = GpuCase(wl, dev, api.INVARIANT)
    kv_bytes = wl.kv_bytes()

    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    # the step as a user runs it (no events between its kernels), NVML
    # sampling the clocks while it runs
    clocks = ClockSampler(local)
    rec = measure(case, peak, peak_kind, args.steps, args.warmup, world, dev, clocks)
    ms_per_step = rec["ms_per_step"]
    value = replica_value(kv_bytes, world, ms_per_step) / 1e9
    e2e_ms, h2d, d2h, e2e_same = e2e_steps(case, max(20, args.steps // 4), args.warmup)
    e2e_ms = max_over_ranks(e2e_ms, dev)

    if rank != 0:
        return

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "math": "fp32",
        "data": "synthetic",
        "config": {
            "workload": wl.name, "rows": wl.B, "H_q": wl.H_q, "H_kv": wl.H_kv,
            "head_dim": wl.D_qk, "layout": wl.layout, "page_size": wl.page_size,
            "kv_bytes_per_step": kv_bytes, "policy": "invariant", "l2": rec["l2"],
            "parallelism": f"replicas x{world}",
        },
        "rows_per_s": rec["rows_per_s"],
        "hbm_frac_of_" + peak_kind: round(value / world / peak, 4),
        "balanced": rec["balanced"],
        "roofline": rec["roofline"],
        "e2e": {"value": round(replica_value(kv_bytes, world, e2e_ms) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "resident": "KV cache",
                "api": "decode_attn_forward",
                "staging": "inputs in one pinned buffer, outputs in one device buffer: "
                           "one copy each way per step",
                "result_equals_device_step": e2e_same},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks.summary(),
    }
    if "roofline_tensor" in rec:
        line["roofline_tensor"] = rec["roofline_tensor"]
    if not args.no_extra:
        extra = {}
        for name in ("gqa_paged", "mla_sparse", "mla_sparse_fp8", "gqa16_paged", "gqa16_paged_fp8",
                     "gqa16_paged_nvfp4", "tiny",
                     "gqa_paged_fp8",
                     "long_context_fp8", "gqa_paged_nvfp4", "long_context_nvfp4",
                     "long_context"):
            if name == args.workload:
                continue
            w2 = build_workload(name)
            c2 = GpuCase(w2, dev, api.INVARIANT)
            n = 40 if name.startswith("long_context") else 200
            extra[w2.name] = measure(c2, peak, peak_kind, n, 5)
            del c2, w2
            torch.cuda.empty_cache()
        line["other_workloads"] = extra
        line["invariance_sweep"] = invariance_sweep(api)
        line["nvfp4_mm"] = nvfp4_section(api, peak)
        gbs, rps, done, dt = cpu_oracle_rate(wl, budget_s=12.0, cycle=True)
        line["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": _CORES,
                                "cpu": cpu_model(), "kind": "oracle",
                                "rows_per_s": round(rps, 3),
                                "sample": f"{done} rows of {wl.name} (its {wl.B} rows in "
                                          f"turn), all heads, {dt:.1f} s, numpy fp64"}
    print(json.dumps(line), flush=True)


def reference_arm(args, rank, world):
    """The oracle as it stands, on host cores, on the same workload: each step
    is a bounded sample of it -- the query heads of one KV head of one row,
    cycling over rows and KV heads."""
    if rank != 0:
        return
    wl = build_workload(args.workload)
    for i in range(args.warmup):
        cpu_oracle_rate(wl, budget_s=0.0, max_rows=1, group=i % wl.H_kv, first_row=i)
    rates = []
    t0 = time.perf_counter()
    for i in range(args.steps):
        gbs, _, _, _ = cpu_oracle_rate(wl, budget_s=0.0, max_rows=1, group=i % wl.H_kv,
                                       first_row=i // wl.H_kv)
        rates.append(gbs)
    elapsed = time.perf_counter() - t0
    value = statistics.median(rates)
    sample = (f"per step: query heads of one KV head of one row of {wl.name} "
              f"(1/{wl.H_kv} of a row), numpy fp64")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * elapsed / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "rows": wl.B, "policy": "oracle (exact softmax)"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": _CORES,
                         "cpu": cpu_model(), "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
