#!/usr/bin/env python3
"""Benchmark of one decode step of the stack-wide paged-FP8 attention path.

One step = gk_kv_append (RoPE(k), E4M3 quantise, packed-K / plain-V scatter for
every layer) + gk_decode_attn_stack (GQA decode attention over every layer
through the full or trimmed sliding-window block table), on synthetic inputs
from gk_inputs with the KV cache resident in HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl gk|reference]

Prints ONE JSON line (rank 0).  `value` is layer*seq/s (layers x active rows
per step / step time) over all ranks; `e2e` is the same metric with the step's
inputs copied from pinned host memory and the output copied back inside the
timed region; `roofline` is for the attention call (planner + persistent
kernel): algorithmic bytes (KV bytes the step must read, counted exactly from
the context lengths, plus q and out) / its CUDA-event duration, against the
measured HBM copy bandwidth.  On the default workload at one GPU the line also
carries `per_config`: the same figures for every other workload of the
measurement, each timed in the same run.  `--impl reference` times the oracle
(plain C) on whole rows of the same workload on the host cores.
Multi-GPU: `--gpus N` starts N replicas itself (torch.distributed.run, one
process per GPU) unless it already runs under a launcher with WORLD_SIZE = N.
Every rank runs an independent replica (no collective on the data path, no
NCCL); the timing reduction (max over ranks of the elapsed time, sum of the
units) goes through a gloo group on the host.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import gk_inputs as gi  # noqa: E402

METRIC = "decode-attn layer·seq/s and achieved HBM GB/s (% of roofline), 1 GB300"
UNIT = "layer·seq/s"
DEFAULT_WORKLOAD = "gptoss_b64"
NOMINAL_HBM_GBS = 7900.0   # GB300 HBM3e, nominal (context beside the measured peak)
ATTN_SOURCES = ["paged_fp8_kv_gk_gb300/csrc/gk_kernels.cu", "paged_fp8_kv_gk_gb300/csrc/gk_device.cuh",
                "paged_fp8_kv_gk_gb300/csrc/gk_internal.h"]


# ------------------------------------------------------------------ distributed
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), ws


def dist_init(backend: str = "gloo"):
    import torch.distributed as dist
    rank, _, ws = dist_env()
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend, rank=rank, world_size=ws)
    return dist if ws > 1 else None


def reduce_timing(local_ms: float, local_units: float, dist=None, device=None):
    """(max elapsed ms over ranks, total units over ranks), on the host (gloo)."""
    if dist is None:
        return local_ms, local_units
    import torch
    t = torch.tensor([local_ms], dtype=torch.float64)
    u = torch.tensor([local_units], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def launch_replicas(gpus: int, argv) -> int:
    """--gpus N outside a launcher: run this script as N ranks on this node
    (torch.distributed.run, rendezvous on 127.0.0.1) and return its exit code;
    None when this process is already a rank (WORLD_SIZE set) or N == 1."""
    if "WORLD_SIZE" in os.environ:
        ws = int(os.environ["WORLD_SIZE"])
        if ws != gpus:
            raise SystemExit(f"--gpus {gpus} but WORLD_SIZE={ws}: launch one rank per GPU")
        return None
    if gpus == 1:
        return None
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={gpus}", "--master-addr", "127.0.0.1", f"--master-port={port}",
           os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


# ------------------------------------------------------------------ helpers
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def attn_source_hash() -> str:
    """Hash of the attention kernel's sources with comments and blank space
    removed (an edit of a comment is not a change of the kernel)."""
    import re
    h = hashlib.sha256()
    for rel in ATTN_SOURCES:
        with open(os.path.join(ROOT, rel)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update("".join(text.split()).encode())
    return h.hexdigest()[:16]


# DRAM traffic of the attention kernel is captured on a reduced case of each
# workload (same per-row shape, a few GB of KV, larger than L2) and scaled to
# the full workload by the ratio of algorithmic bytes per launch.
TRAFFIC_CASES = {"gptoss_b64": "gptoss_b16", "swa_b512": "swa_b128", "long_ctx": "long_b1",
                 "ragged_b256": "ragged_b24", "gk120b_rank_b64": "gk120b_rank_b64"}


def traffic_command(case: str) -> str:
    return ("ncu --metrics gpu__time_duration.sum,dram__bytes_read.sum,dram__bytes_write.sum "
            "--clock-control none -k regex:attn_kernel -s 3 -c 3 --csv --log-file launches.csv "
            f"python bench.py --workload {case} --steps 3 --warmup 3 --no-cpu-baseline "
            "--no-per-config")


def alg_bytes(w, c) -> int:
    """Algorithmic bytes of one attention launch: KV read (exact) + q + out."""
    return gi.kv_bytes_read(w, c) + gi.qo_bytes(w, c)


def recorded_traffic(w, c):
    """DRAM bytes per attention launch of workload w, from the committed ncu
    capture of its reduced case scaled by algorithmic bytes, if that capture
    was taken on the current kernel source; else None.  Returns
    (bytes, reduced case, scale)."""
    p = os.path.join(ROOT, "profiles", "attn_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    case = TRAFFIC_CASES.get(w.name, w.name)
    e = d.get(case)
    if not e or e.get("kernel_src_sha") != attn_source_hash():
        return None
    scale = alg_bytes(w, c) / e["alg_bytes_per_launch"]
    return int(round(e["dram_bytes_per_launch"] * scale)), case, scale


def record_traffic(case: str, csv_path: str, out_path: str = None) -> dict:
    """Average DRAM bytes per attention launch from an ncu launch list of this
    bench on the reduced case `case` (traffic_command(case)) into
    profiles/attn_traffic.json, with the case's algorithmic bytes per launch
    and the current kernel source hash."""
    import csv
    vals = {}
    with open(csv_path) as f:
        rows = [r for r in csv.reader(f) if len(r) > 5]
    hdr = {k: i for i, k in enumerate(rows[0])}
    for r in rows[1:]:
        if "attn_kernel" not in r[hdr["Kernel Name"]]:
            continue
        v = float(r[hdr["Metric Value"]].replace(",", ""))
        vals.setdefault(r[hdr["Metric Name"]], []).append(v)
    rd = statistics.fmean(vals["dram__bytes_read.sum"])
    wr = statistics.fmean(vals["dram__bytes_write.sum"])
    w = gi.get(case)
    c = gi.make_control(w)
    entry = {"kernel_src_sha": attn_source_hash(), "dram_bytes_per_launch": int(rd + wr),
             "dram_read_bytes": int(rd), "dram_write_bytes": int(wr),
             "alg_bytes_per_launch": alg_bytes(w, c),
             "launches_averaged": len(vals["dram__bytes_read.sum"]),
             "avg_launch_ns_under_ncu": round(statistics.fmean(vals["gpu__time_duration.sum"]), 1),
             "command": traffic_command(case)}
    p = out_path or os.path.join(ROOT, "profiles", "attn_traffic.json")
    d = {}
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
    d[case] = entry
    with open(p, "w") as f:
        json.dump(d, f, indent=1)
        f.write("\n")
    return entry


def device_selector(dev) -> str:
    """The GPU of torch device `dev` as nvidia-smi / NVML name it (UUID, else
    PCI bus id; NVML ignores CUDA_VISIBLE_DEVICES, so an index would not do)."""
    import torch
    pr = torch.cuda.get_device_properties(dev)
    u = getattr(pr, "uuid", None)
    if u is not None:
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    if hasattr(pr, "pci_bus_id"):
        return f"{pr.pci_domain_id:08X}:{pr.pci_bus_id:02X}:{pr.pci_device_id:02X}.0"
    return str(dev.index or 0)


class NvmlClockSampler:
    """SM clock, power and clock-event reasons read through NVML (the driver's
    libnvidia-ml, read-only queries) every `period_s` on a host thread; only
    the samples taken between mark_begin and mark_end count.  Fine enough to
    put several samples inside a timed region of a few milliseconds."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, selector: str, period_s: float = 0.002):
        import ctypes
        import threading
        self.period = period_s
        self.rows = []
        self.t0 = self.t1 = None
        L = ctypes.CDLL("libnvidia-ml.so.1")
        if L.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.L = L
        self.h = ctypes.c_void_p()
        if selector.startswith("GPU-"):
            rc = L.nvmlDeviceGetHandleByUUID(selector.encode(), ctypes.byref(self.h))
        else:
            rc = L.nvmlDeviceGetHandleByPciBusId_v2(selector.encode(), ctypes.byref(self.h))
        if rc != 0:
            raise OSError(f"no NVML handle for {selector}")
        self.reasons_fn = getattr(L, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            L.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        L.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))
        self.max_mhz = float(mx.value)
        self.stop_ev = threading.Event()
        self.thread = threading.Thread(target=self._loop, daemon=True)

    def _loop(self):
        import ctypes
        clk, rs, pw = ctypes.c_uint(), ctypes.c_ulonglong(), ctypes.c_uint()
        while not self.stop_ev.is_set():
            t = time.perf_counter()
            self.L.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk))
            self.reasons_fn(self.h, ctypes.byref(rs))
            self.L.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(pw))
            self.rows.append((t, float(clk.value), int(rs.value), pw.value / 1000.0))
            time.sleep(self.period)

    def start(self):
        self.thread.start()
        time.sleep(0.05)

    def mark_begin(self):
        self.t0 = time.perf_counter()

    def mark_end(self):
        self.t1 = time.perf_counter()

    def stop(self):
        time.sleep(0.02)
        self.stop_ev.set()
        self.thread.join(timeout=5)
        self.L.nvmlShutdown()
        inside = [r for r in self.rows if self.t0 is not None and self.t0 <= r[0] <= (self.t1 or r[0])]
        use = inside if inside else self.rows
        if not use:
            return None
        reasons = sorted({n for r in use for bit, n in self.REASONS.items() if r[2] & bit})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": self.max_mhz,
                "samples": len(self.rows), "samples_in_timed_region": len(inside),
                "power_w_max": max(r[3] for r in use), "reasons": reasons, "source": "nvml"}


def clock_sampler(dev):
    """NVML sampler for the GPU of `dev`, else the nvidia-smi one."""
    sel = device_selector(dev)
    try:
        return NvmlClockSampler(sel)
    except (OSError, AttributeError):
        return ClockSampler(sel)


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons; only samples whose
    timestamp falls inside the timed region (mark_begin .. mark_end) count."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(prefix="gk_clocks_", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        self.t0 = self.t1 = None

    def mark_begin(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        import datetime
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(parts[1]), float(parts[2]),
                                 [n for n, v in zip(names, parts[4:8]) if v.lower().startswith("active")]))
                except ValueError:
                    continue
        os.unlink(self.path)
        inside = [r for r in rows if self.t0 is not None and self.t0 <= r[0] <= (self.t1 or r[0])]
        use = inside if inside else rows
        if not use:
            return None
        reasons = sorted({n for r in use for n in r[3]})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "samples": len(use), "samples_in_timed_region": len(inside), "reasons": reasons}


def kv_layout_desc(k_layout: str = "packed", kv_form: str = "per_group") -> str:
    form = ("per-group buffers [2,nb,kv,B,D]" if kv_form == "per_group"
            else "stacked K_cache/V_cache [G,nb,kv,B,D]")
    k = "K packed [..,B/2,D,2]" if k_layout == "packed" else "K unpacked [..,B,D]"
    return f"{form}, {k}, E4M3"


def workload_config(w, c, kv_layout: str = None):
    kind, _, arg = w.lengths.partition(":")
    return {"workload": w.name, "num_layers": w.num_layers, "batch": w.batch,
            "active_rows": int(c.active.sum()), "q_heads": w.num_q_heads,
            "kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "block_size": w.block_size,
            "window": w.window, "context": f"{kind}:{arg}", "mean_context": float(c.lengths[c.active == 1].mean()),
            "kv_layout": kv_layout or kv_layout_desc()}


# ------------------------------------------------------------------ CPU baseline (oracle)
def oracle_threads() -> int:
    """Host threads for the oracle timing: the cores this process may use."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


class OracleRows:
    """The oracle (plain C) on whole rows of a workload: one task = row b,
    every layer pair (append + attention, all kv heads).  Row pools are copied
    to host memory before any timing.  The C calls release the GIL, so rows
    run in parallel on host threads (no process is forked)."""

    def __init__(self, w, c, step_host, cache, k_layout: int = 0):
        self.w, self.c, self.host, self.cache, self.k_layout = w, c, step_host, cache, k_layout
        self.pools = {}

    def prepare(self, b: int):
        import torch
        c, cache = self.c, self.cache
        for j in range(self.w.num_layers // 2):
            if (b, j) in self.pools:
                continue
            ids = np.concatenate([np.asarray(c.full_blocks[b], np.int64),
                                  np.asarray(c.swa_blocks[b], np.int64)])
            idx = torch.as_tensor(ids, device=cache[j][0].device)
            self.pools[(b, j)] = (cache[j][0].index_select(0, idx).cpu().numpy().reshape(-1),
                                  cache[j][1].index_select(0, idx).cpu().numpy().reshape(-1))

    def row(self, b: int) -> int:
        import oracle.rows as orows
        for j in range(self.w.num_layers // 2):
            kp, vp = self.pools[(b, j)]
            orows.row_pair_from_pool(self.w, self.c, self.host, kp, vp, j, b,
                                     k_layout=self.k_layout)
        return self.w.num_layers

    def timed(self, rows, threads: int):
        """Wall seconds and layer*seq units for `rows` on `threads` threads."""
        from concurrent.futures import ThreadPoolExecutor
        for b in rows:
            self.prepare(int(b))
        t0 = time.perf_counter()
        if threads == 1:
            units = sum(self.row(int(b)) for b in rows)
        else:
            with ThreadPoolExecutor(max_workers=threads) as ex:
                units = sum(ex.map(self.row, [int(b) for b in rows]))
        return time.perf_counter() - t0, units


def oracle_sample(w, c, step_host, cache, budget_s: float, seed: int = 0, k_layout: int = 0):
    """The cpu_baseline: the oracle on a bounded sample of whole rows, first on
    one thread (one row), then on every host core (enough rows for about
    `budget_s` seconds of CPU work).  Returns a dict for the JSON line."""
    rng = np.random.default_rng(seed)
    rows = [int(b) for b in rng.permutation(np.nonzero(c.active)[0])]
    o = OracleRows(w, c, step_host, cache, k_layout)
    t1, u1 = o.timed(rows[:1], 1)
    T = oracle_threads()
    n = max(T, int(round(budget_s / max(t1, 1e-3))))
    sample = [rows[i % len(rows)] for i in range(1, 1 + n)]
    tT, uT = o.timed(sample, T)
    return {"value": round(uT / tT, 3), "unit": UNIT, "cores": T, "kind": "oracle",
            "single_thread_value": round(u1 / t1, 3),
            "sample": f"{len(sample)} rows x {w.num_layers} layers (all kv heads) on {T} threads, "
                      f"{tT:.1f} s wall; single thread: 1 row, {t1:.1f} s; oracle append + fp64 "
                      f"attention"}


# ------------------------------------------------------------------ end-to-end loop
def run_e2e(gk, shape, inputs, kv, out, ws, stream, dev, K, W, units, dist, fused=False):
    """Time K steps fed from pinned host memory: per step one H2D copy of all
    inputs (packed), the step (gk_decode_step, or gk_kv_append +
    gk_decode_attn_stack), one D2H copy of the output.  Returns (max ms over
    ranks, units over ranks, H2D bytes/step, D2H bytes/step)."""
    import torch
    names = list(inputs)
    offs, off = {}, 0
    for n in names:
        nb = inputs[n].numel() * inputs[n].element_size()
        offs[n] = off
        off += (nb + 255) // 256 * 256
    total = off
    host = torch.empty(total, dtype=torch.uint8).pin_memory()
    for n in names:
        t = inputs[n]
        nb = t.numel() * t.element_size()
        host[offs[n]:offs[n] + nb].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())
    dbuf = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]

    def views(buf):
        v = {}
        for n in names:
            t = inputs[n]
            nb = t.numel() * t.element_size()
            v[n] = buf[offs[n]:offs[n] + nb].view(t.dtype).view(t.shape)
        return v

    dv = [views(b) for b in dbuf]
    outs = [out, torch.empty_like(out)]
    host_out = torch.empty(out.numel() * out.element_size(), dtype=torch.uint8).pin_memory()
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    sh = stream.cuda_stream

    def step(k):
        i = k % 2
        d = dv[i]
        if k >= 2:
            s_in.wait_event(ev_done[i])          # kernels of step k-2 are done with buffer i
        with torch.cuda.stream(s_in):
            dbuf[i].copy_(host, non_blocking=True)
            ev_in[i].record(s_in)
        stream.wait_event(ev_in[i])
        if k >= 2:
            stream.wait_event(ev_out[i])         # output i of step k-2 has been read back
        if fused:
            gk.gk_decode_step(shape, d["q"], d["k_new"], d["v_new"], d["cos"], d["sin"],
                              d["k_scale"], d["v_scale"], d["upd_full"], d["upd_swa"],
                              d["bt_full"], d["bt_swa"], d["pos"], d["pos_w"], d["active"], kv,
                              outs[i], None, ws, stream=sh)
        else:
            gk.gk_kv_append(shape, d["k_new"], d["v_new"], d["cos"], d["sin"], d["k_scale"],
                            d["v_scale"], d["upd_full"], d["upd_swa"], d["active"], kv, stream=sh)
            gk.gk_decode_attn_stack(shape, d["q"], kv, d["k_scale"], d["v_scale"], d["cos"],
                                    d["sin"], d["bt_full"], d["bt_swa"], d["pos"], d["pos_w"],
                                    d["active"], outs[i], None, ws, stream=sh)
        ev_done[i].record(stream)
        s_out.wait_event(ev_done[i])
        with torch.cuda.stream(s_out):
            host_out.copy_(outs[i].view(-1).view(torch.uint8), non_blocking=True)
            ev_out[i].record(s_out)

    for k in range(W):
        step(k)
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for k in range(K):
        step(k)
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    ms, u = reduce_timing(e0.elapsed_time(e1), units * K, dist, dev)
    return ms, u, total, host_out.numel()


# ------------------------------------------------------------------ main arms
# Workloads reported beside the headline one, each measured in the same run.
PER_CONFIG = ["tiny", "long_ctx", "ragged_b256", "swa_b512", "gk120b_rank_b64"]


def measure_step(args, name, dev, dist, with_clocks=False, with_oracle=False):
    """Time one workload: whole steps (append + attention, or gk_decode_step),
    the attention call alone (roofline), the append alone, and the
    end-to-end loop from pinned host memory.  Returns the JSON fields."""
    import torch
    import paged_fp8_kv_gk_gb300 as gk
    rank, local_rank, world = dist_env()
    w = gi.get(name)
    c = gi.make_control(w)
    st = gi.make_step(w, dev)
    cache = gi.make_cache(w, c, dev)
    shape = gk.Shape.make(**gi.shape_dict(w, c))
    t = lambda a, dt: torch.as_tensor(np.ascontiguousarray(a)).to(dev, dt)  # noqa: E731
    ctl = dict(cos=t(c.cos, torch.float32), sin=t(c.sin, torch.float32),
               k_scale=t(c.k_scale, torch.float32), v_scale=t(c.v_scale, torch.float32),
               bt_full=t(c.bt_full, torch.int32), bt_swa=t(c.bt_swa, torch.int32),
               pos=t(c.pos, torch.int32), pos_w=t(c.pos_w, torch.int32),
               upd_full=t(c.upd_full, torch.int32), upd_swa=t(c.upd_swa, torch.int32),
               active=t(c.active, torch.uint8))
    q, k_new, v_new = st["q"].contiguous(), st["k_new"].contiguous(), st["v_new"].contiguous()
    k_layout = gk.GK_K_PLAIN if args.k_layout == "plain" else gk.GK_K_PACKED
    if args.kv_form == "stacked":
        # K_cache / V_cache with a leading group axis, one allocation each
        kst = torch.stack([b[0] for b in cache])
        vst = torch.stack([b[1] for b in cache])
        cache = [(kst[j], vst[j]) for j in range(len(cache))]  # the same bytes, per group
        kc = kst
        if k_layout == gk.GK_K_PACKED:
            G, nbk, kvh, Bk, Dk = kst.shape
            kc = kst.view(G, nbk, kvh, Bk // 2, Dk, 2)
        kv = gk.kv_stacked(kc, vst)
    else:
        kv = gk.kv_from_group_buffers(cache, k_layout)
    out = torch.empty(w.num_layers, w.batch, w.num_q_heads, w.head_dim, dtype=torch.bfloat16,
                      device=dev)
    if args.ws_min:   # smallest workspace: no split-KV (profiling the unsplit stage loop)
        ws = torch.empty(gk.gk_attn_workspace_min_bytes(shape), dtype=torch.uint8, device=dev)
    else:
        ws = gk.new_workspace(shape, dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    def append():
        gk.gk_kv_append(shape, k_new, v_new, ctl["cos"], ctl["sin"], ctl["k_scale"],
                        ctl["v_scale"], ctl["upd_full"], ctl["upd_swa"], ctl["active"], kv,
                        stream=sh)

    def attention():
        gk.gk_decode_attn_stack(shape, q, kv, ctl["k_scale"], ctl["v_scale"], ctl["cos"],
                                ctl["sin"], ctl["bt_full"], ctl["bt_swa"], ctl["pos"],
                                ctl["pos_w"], ctl["active"], out, None, ws, stream=sh)

    def fused_step():
        gk.gk_decode_step(shape, q, k_new, v_new, ctl["cos"], ctl["sin"], ctl["k_scale"],
                          ctl["v_scale"], ctl["upd_full"], ctl["upd_swa"], ctl["bt_full"],
                          ctl["bt_swa"], ctl["pos"], ctl["pos_w"], ctl["active"], kv, out,
                          None, ws, stream=sh)

    if args.step == "fused":
        def one_step():
            fused_step()
    else:
        def one_step():
            append()
            attention()

    if args.graph:
        # the whole step captured once (on a side stream: the legacy default
        # stream cannot be captured) and replayed on the timing stream
        one_step()                       # device setup happens outside the capture
        torch.cuda.synchronize(dev)
        cap = torch.cuda.Stream(dev)
        sh = cap.cuda_stream
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            one_step()
        sh = stream.cuda_stream

        def one_step():
            graph.replay()

    K, W = args.steps, args.warmup
    for _ in range(W):
        one_step()
    torch.cuda.synchronize(dev)
    if gk.gk_read_device_error() != 0:
        raise RuntimeError(f"{name}: device error word set during warm-up")

    # L2: a step whose KV is not well above the L2 size would find part of it
    # still cached from the step before; such steps are timed one by one with
    # a write of twice the L2 size between them, outside the timed events
    kv_bytes = gi.kv_bytes_read(w, c)
    l2_bytes = int(torch.cuda.get_device_properties(dev).L2_cache_size)
    flush = args.flush_l2 == "on" or (args.flush_l2 == "auto" and kv_bytes < 2 * l2_bytes)
    flush_buf = torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev) if flush else None
    if flush:
        l2_note = (f"L2 flushed before every timed step ({2 * l2_bytes / 1e6:.0f} MB write, outside "
                   f"the events; {kv_bytes / 1e9:.3f} GB KV read per step; e2e unflushed)")
    elif kv_bytes >= 2 * l2_bytes:
        l2_note = f"inputs larger than L2: {kv_bytes / 1e9:.2f} GB KV read per step"
    else:
        l2_note = (f"L2 not flushed (--flush-l2 off): {kv_bytes / 1e9:.3f} GB KV read per step, "
                   f"under twice the L2 size")

    def l2_flush(k):
        if flush:
            flush_buf.fill_(k & 0xff)

    # ---- timed loop 1: whole steps (append + attention), events only at the
    # two ends so that nothing sits between the kernels of a step
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    clocks = clock_sampler(dev) if with_clocks else None
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    if clocks:
        clocks.start()
        clocks.mark_begin()
    if flush:
        s0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        s1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        for k in range(K):
            l2_flush(k)
            s0[k].record(stream)
            one_step()
            s1[k].record(stream)
    else:
        ev0.record(stream)
        for k in range(K):
            one_step()
        ev1.record(stream)
    torch.cuda.synchronize(dev)
    if clocks:
        clocks.mark_end()
    clk = clocks.stop() if clocks else None
    if dist:
        dist.barrier()
    if flush:
        elapsed_ms = sum(s0[k].elapsed_time(s1[k]) for k in range(K))
    else:
        elapsed_ms = ev0.elapsed_time(ev1)

    # ---- timed loop 2: the attention call (planner + persistent kernel) alone,
    # an event pair around every launch, for the roofline of the dominant kernel
    a0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    a1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for k in range(K):
        l2_flush(k)
        a0[k].record(stream)
        attention()
        a1[k].record(stream)
    torch.cuda.synchronize(dev)
    attn_all = [a0[k].elapsed_time(a1[k]) for k in range(K)]
    attn_ms = statistics.fmean(attn_all)
    attn_med = statistics.median(attn_all)
    # the append alone, for the record
    for k in range(K):
        l2_flush(k)
        a0[k].record(stream)
        append()
        a1[k].record(stream)
    torch.cuda.synchronize(dev)
    append_ms = statistics.fmean(a0[k].elapsed_time(a1[k]) for k in range(K))
    # the other step form, for the record (gk_kv_append + gk_decode_attn_stack
    # beside gk_decode_step, or the reverse), timed like timed loop 1
    def other_step():
        if args.step == "fused":
            append()
            attention()
        else:
            fused_step()
    for _ in range(W):
        other_step()
    torch.cuda.synchronize(dev)
    if flush:
        for k in range(K):
            l2_flush(k)
            a0[k].record(stream)
            other_step()
            a1[k].record(stream)
        torch.cuda.synchronize(dev)
        other_ms = sum(a0[k].elapsed_time(a1[k]) for k in range(K)) / K
    else:
        ev0.record(stream)
        for k in range(K):
            other_step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        other_ms = ev0.elapsed_time(ev1) / K
    units = gi.layer_seqs(w, c)
    max_ms, total_units = reduce_timing(elapsed_ms, units * K, dist, dev)
    value = total_units / (max_ms / 1e3)

    # ---- end to end: every step's inputs copied from pinned host memory (one
    # packed staging copy) and its output copied back, double-buffered on two
    # copy streams so that step k+1's upload and step k's download overlap
    # step k's kernels.
    e2e_ms, e2e_units, h2d, d2h = run_e2e(gk, shape, dict(q=q, k_new=k_new, v_new=v_new, **ctl),
                                          kv, out, ws, stream, dev, K, W, units, dist,
                                          fused=args.step == "fused")
    if gk.gk_read_device_error() != 0:
        raise RuntimeError(f"{name}: device error word set during the timed region")

    # ---- roofline of the attention call
    ab = alg_bytes(w, c)
    peak, peak_kind = measured_peaks()
    achieved = ab / (attn_ms / 1e3) / 1e9
    tr = recorded_traffic(w, c)
    res = {
        "value": round(value, 1), "ms_per_step": round(max_ms / K, 4),
        "config": workload_config(w, c, kv_layout_desc(args.k_layout, args.kv_form)),
        "l2": l2_note,
        "attn_ms": round(attn_ms, 4), "attn_ms_median": round(attn_med, 4),
        "append_ms": round(append_ms, 4), "achieved_GBps": round(achieved, 1),
        "other_step": {"form": ("gk_kv_append + gk_decode_attn_stack" if args.step == "fused"
                                else "gk_decode_step"), "ms_per_step": round(other_ms, 4)},
        "kv_bytes_per_step": kv_bytes, "qo_bytes_per_step": gi.qo_bytes(w, c),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": tr[0] if tr else None,
                     "traffic_source": (f"ncu dram__bytes_read.sum + dram__bytes_write.sum on "
                                        f"{tr[1]}, scaled x{tr[2]:.4f} by algorithmic bytes"
                                        if tr else None),
                     "peak_source": peak_kind, "peak_nominal": NOMINAL_HBM_GBS,
                     "frac_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                     "kernel": "gk_decode_attn_stack (plan_kernel + attn_kernel)",
                     "alg_bytes_per_launch": ab},
        "e2e": {"value": round(e2e_units / (e2e_ms / 1e3), 1), "unit": UNIT,
                "ms_per_step": round(e2e_ms / K, 4), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "clocks": clk,
        # the combine kernel runs when the workspace holds partial records:
        # the recommended workspace does once a row may exceed 512 keys
        "combine_launched": int(not args.ws_min and c.max_blocks_full * w.block_size > 512),
    }
    if with_oracle:
        host = {k: gi.bf16_bits(v) for k, v in st.items()}
        res["cpu_baseline"] = oracle_sample(w, c, host, cache, args.cpu_budget, k_layout=k_layout)
    return res


def run_gk(args):
    import torch
    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    dist = dist_init("gloo")
    dev = torch.device("cuda", local_rank)
    K, W = args.steps, args.warmup
    head = measure_step(args, args.workload, dev, dist, with_clocks=True,
                        with_oracle=rank == 0 and world == 1 and not args.no_cpu_baseline)
    line = {
        "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "precision": "KV E4M3 codes; q/out bf16; QK^T and PV on f16 tensor-core MMA with fp32 "
                     "accumulation; fp32 online softmax",
        "data": "synthetic (seeded gk_inputs workload)",
        "impl": "gk",
        "step_form": ("gk_decode_step" if args.step == "fused" else
                      "gk_kv_append + gk_decode_attn_stack") + (" (CUDA graph)" if args.graph else ""),
        # per timed step: (plan + append) + attention [+ split-KV combine] for
        # gk_decode_step; append + plan + attention [+ combine] for the two calls
        "gpu_launches": ((2 if args.step == "fused" else 3) + head["combine_launched"]) * K,
    }
    line.update({k: v for k, v in head.items() if k != "combine_launched"})
    if world == 1 and not args.no_per_config and args.workload == DEFAULT_WORKLOAD:
        per = {}
        for name in PER_CONFIG:
            r = measure_step(args, name, dev, dist)
            per[name] = {"value": r["value"], "unit": UNIT, "ms_per_step": r["ms_per_step"],
                         "attn_ms": r["attn_ms"], "achieved_GBps": r["achieved_GBps"],
                         "frac": r["roofline"]["frac"],
                         "frac_nominal": r["roofline"]["frac_nominal"],
                         "traffic": r["roofline"]["traffic"], "e2e": r["e2e"]["value"],
                         "other_step_ms": r["other_step"]["ms_per_step"],
                         "alg_bytes_per_launch": r["roofline"]["alg_bytes_per_launch"],
                         "config": r["config"], "l2": r["l2"]}
            torch.cuda.empty_cache()
        line["per_config"] = per
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def run_ingest(args):
    """The DI landing copy (gk_kv_ingest) on its own: every block a batch of
    prompts sends (both engines at N - 1) landed on a fresh decode cache, per
    step.  value = bytes moved (read + write) per second, against the copy
    bandwidth; e2e = the same landing read straight from pinned host memory."""
    import torch
    import paged_fp8_kv_gk_gb300 as gk
    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    dist = dist_init("gloo")
    dev = torch.device("cuda", local_rank)
    w = gi.get(args.workload)
    c = gi.make_control(w)
    truth = gi.make_cache(w, c, dev)
    dr, db, src = gi.make_landing(w, c, truth)
    del truth
    cache = [torch.zeros(2, c.num_blocks, w.num_kv_heads, w.block_size, w.head_dim,
                         dtype=torch.uint8, device=dev) for _ in range(w.num_layers // 2)]
    kv = gk.kv_from_group_buffers(cache)
    lk, lv = gk.layer_binding(kv, w.num_layers)
    regions = gk.gk_kv_regions(gk.Shape.make(**gi.shape_dict(w, c)), lk, lv)
    dr_t = torch.as_tensor(dr, device=dev)
    db_t = torch.as_tensor(db, device=dev)
    landed = src.numel()
    stream = torch.cuda.current_stream(dev)

    def timed(source, K, W):
        for _ in range(W):
            gk.gk_kv_ingest(regions, dr_t, db_t, source, stream=stream)
        torch.cuda.synchronize(dev)
        if gk.gk_read_device_error() != 0:
            raise RuntimeError("device error word set during warm-up")
        e0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        e1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        if dist:
            dist.barrier()
        torch.cuda.synchronize(dev)
        for k in range(K):
            e0[k].record(stream)
            gk.gk_kv_ingest(regions, dr_t, db_t, source, stream=stream)
            e1[k].record(stream)
        torch.cuda.synchronize(dev)
        return [e0[k].elapsed_time(e1[k]) for k in range(K)]

    K, W = args.steps, args.warmup
    clocks = clock_sampler(dev)
    clocks.start()
    clocks.mark_begin()
    per = timed(src, K, W)
    clocks.mark_end()
    clk = clocks.stop()
    ms = statistics.fmean(per)
    max_ms, units = reduce_timing(sum(per), 2 * landed * K, dist, dev)
    value = units / (max_ms / 1e3) / 1e9
    host = src.cpu().pin_memory()
    per_h = timed(host, max(3, K // 4), 2)
    e2e_ms = statistics.fmean(per_h)
    peak, peak_kind = measured_peaks()
    achieved = 2 * landed / (ms / 1e3) / 1e9
    line = {
        "metric": "DI KV landing bandwidth (read + write bytes/s), 1 GB300", "value": round(value, 1),
        "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic (seeded gk_inputs workload)",
        "config": dict(workload_config(w, c), op="gk_kv_ingest", descriptors=int(dr.size),
                       block_len=int(src.shape[1])),
        "l2": f"inputs larger than L2: {landed / 1e9:.2f} GB landed per step",
        "impl": "gk",
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": None, "peak_source": peak_kind,
                     "kernel": "ingest_kernel", "alg_bytes_per_launch": 2 * landed},
        "e2e": {"value": round(landed / (e2e_ms / 1e3) / 1e9, 1), "unit": "GB/s landed",
                "source": "pinned host memory read by the kernel", "h2d_bytes_per_step": landed,
                "d2h_bytes_per_step": 0},
        "gpu_launches": K,
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def run_reference(args):
    """The oracle timed on the host cores: each step is one whole row of the
    workload (every layer pair, every kv head); the steps run on every host
    core (threads; the C calls release the GIL)."""
    import torch
    rank, local_rank, world = dist_env()
    if rank != 0:
        return
    w = gi.get(args.workload)
    c = gi.make_control(w)
    dev = torch.device("cuda", local_rank) if torch.cuda.is_available() else torch.device("cpu")
    st = gi.make_step(w, dev)
    cache = gi.make_cache(w, c, dev)
    host = {k: gi.bf16_bits(v) for k, v in st.items()}
    rng = np.random.default_rng(7)
    rows = [int(b) for b in rng.permutation(np.nonzero(c.active)[0])]
    o = OracleRows(w, c, host, cache)
    T = oracle_threads()
    seq = [rows[s % len(rows)] for s in range(args.warmup + args.steps)]
    if args.warmup:
        o.timed(seq[:args.warmup], T)
    wall, units = o.timed(seq[args.warmup:], T)
    value = units / wall
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * wall / args.steps, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded gk_inputs workload)",
        "config": workload_config(w, c, kv_layout_desc(args.k_layout, args.kv_form)),
        "l2": "host memory (the oracle runs on the host cores)", "impl": "reference",
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": T, "kind": "oracle",
                         "sample": f"each step one row x {w.num_layers} layers (all kv heads): "
                                   f"oracle append + fp64 attention; steps spread over {T} "
                                   f"threads"},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=None,
                    help=f"default {DEFAULT_WORKLOAD} (--op step), di_ingest_b16 (--op ingest)")
    ap.add_argument("--op", choices=["step", "ingest"], default="step",
                    help="step: the decode step (headline); ingest: the DI landing copy alone")
    ap.add_argument("--impl", choices=["gk", "reference"], default="gk")
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle CPU time for the cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="measure the headline workload only (no per_config block)")
    ap.add_argument("--step", choices=["split", "fused"], default="fused",
                    help="fused: gk_decode_step (the append in the planner's launch; the default, "
                         "measured faster); split: gk_kv_append + gk_decode_attn_stack")
    ap.add_argument("--k-layout", choices=["packed", "plain"], default="packed",
                    help="K through the packed view (the page's layout) or unpacked like V")
    ap.add_argument("--kv-form", choices=["per_group", "stacked"], default="per_group",
                    help="per-group K/V buffers or stacked K_cache/V_cache")
    ap.add_argument("--graph", action="store_true",
                    help="time the step as one captured CUDA graph replayed per step")
    ap.add_argument("--record-traffic", metavar="LAUNCHES_CSV", default=None,
                    help="store the attention kernel's DRAM bytes per launch from an ncu launch "
                         "list of the reduced case --workload (see traffic_command) into "
                         "profiles/attn_traffic.json, then exit")
    ap.add_argument("--flush-l2", choices=["auto", "on", "off"], default="auto",
                    help="write twice the L2 size before every timed step (auto: when the KV "
                         "read per step is under twice the L2 size)")
    ap.add_argument("--ws-min", action="store_true",
                    help="use the minimum attention workspace (no split-KV chunks)")
    args = ap.parse_args(argv)
    rc = launch_replicas(args.gpus, sys.argv[1:] if argv is None else list(argv))
    if rc is not None:
        sys.exit(rc)
    if args.record_traffic:
        print(json.dumps(record_traffic(args.workload or DEFAULT_WORKLOAD, args.record_traffic)))
        return
    if args.workload is None:
        args.workload = "di_ingest_b16" if args.op == "ingest" else DEFAULT_WORKLOAD
    if args.op == "ingest":
        if args.impl == "reference":
            raise SystemExit("--op ingest has no reference arm")
        run_ingest(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gk(args)


if __name__ == "__main__":
    main()
