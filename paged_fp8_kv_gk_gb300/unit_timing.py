"""Per-unit timing of the attention kernel (diagnostic; needs a CUDA GPU).

Builds and loads the diagnostic variant of the library (GK_PROBE_UNITS=1: the
same kernels with globaltimer stamps; the product libgk.so has none), runs the
attention call of a seeded workload a few times and prints, per unit kind
(full-layer chunk, sliding-window unit), a least-squares fit of a unit's
consumer time against its number of 32-key stages: the intercept is the fixed
cost of a unit (descriptor, q prologue, epilogue, split partials and merge),
the slope the time of one stage.  It also reports the share of time the warps
spent waiting on stage barriers (staged data not yet there).  The stamps cost a
few instructions per stage, so absolute times run a little slow.

    python -m paged_fp8_kv_gk_gb300.unit_timing gptoss_b64 swa_b512 long_ctx

Run from the repository root (the workloads come from gk_inputs).
"""
from __future__ import annotations

import ctypes
import json
import sys

import numpy as np

PROBE_WARPS, PROBE_UNITS = 4096, 64


def measure(name: str, warmup: int = 5) -> dict:
    import torch

    import gk_inputs as gi
    import paged_fp8_kv_gk_gb300 as gk

    dev = torch.device("cuda", 0)
    w = gi.get(name)
    c = gi.make_control(w)
    st = gi.make_step(w, dev)
    cache = gi.make_cache(w, c, dev)
    shape = gk.Shape.make(**gi.shape_dict(w, c))
    t = lambda a, dt: torch.as_tensor(np.ascontiguousarray(a)).to(dev, dt)  # noqa: E731
    ks, vs = t(c.k_scale, torch.float32), t(c.v_scale, torch.float32)
    cos, sin = t(c.cos, torch.float32), t(c.sin, torch.float32)
    bt_full, bt_swa = t(c.bt_full, torch.int32), t(c.bt_swa, torch.int32)
    pos, pos_w, active = t(c.pos, torch.int32), t(c.pos_w, torch.int32), t(c.active, torch.uint8)
    kv = gk.kv_from_group_buffers(cache, gk.GK_K_PACKED)
    out = torch.empty(w.num_layers, w.batch, w.num_q_heads, w.head_dim, dtype=torch.bfloat16,
                      device=dev)
    ws = gk.new_workspace(shape, dev)
    q = st["q"].contiguous()
    for _ in range(warmup + 1):
        gk.gk_decode_attn_stack(shape, q, kv, ks, vs, cos, sin, bt_full, bt_swa, pos, pos_w,
                                active, out, None, ws)
    torch.cuda.synchronize(dev)
    if gk.gk_read_device_error() != 0:
        raise RuntimeError("device error word set")

    L = gk.lib()
    L.gk_probe_units_read.restype = ctypes.c_int
    L.gk_probe_units_read.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                      ctypes.c_size_t]
    units = np.zeros((PROBE_WARPS, PROBE_UNITS, 4), np.uint64)
    warps = np.zeros((PROBE_WARPS, 2), np.uint64)
    if L.gk_probe_units_read(units.ctypes.data, units.nbytes, warps.ctypes.data, warps.nbytes):
        raise RuntimeError("gk_probe_units_read failed")
    nw = torch.cuda.get_device_properties(dev).multi_processor_count * 16
    units, warps = units[:nw].astype(np.int64), warps[:nw].astype(np.int64)
    count = np.minimum(warps[:, 1], PROBE_UNITS)
    sel = np.arange(PROBE_UNITS)[None, :] < count[:, None]
    u = units[sel]                                   # [n, 4]
    dur = (u[:, 1] - u[:, 0]) / 1e3                  # us, first stage wait .. epilogue end
    wait = u[:, 2] / 1e3
    stages = u[:, 3] & 0xFFFF
    kind = (u[:, 3] >> 16) & 0xF
    nsplit = (u[:, 3] >> 20) & 0xFFF
    res = {"workload": name, "units_timed": int(len(u)), "warps": nw,
           "units_per_warp_median": float(np.median(warps[:, 1])),
           "stage_us": round(float(dur.sum() / stages.sum()), 3),
           "wait_share": round(float(wait.sum() / dur.sum()), 4)}
    for k, label in ((1, "full"), (2, "window")):
        m = kind == k
        if m.sum() < 10:
            continue
        A = np.vstack([np.ones(int(m.sum())), stages[m]]).T
        (a, b), *_ = np.linalg.lstsq(A, dur[m], rcond=None)
        res[label] = {"units": int(m.sum()), "stages_mean": round(float(stages[m].mean()), 2),
                      "us_mean": round(float(dur[m].mean()), 2),
                      "fixed_us": round(float(a), 2), "us_per_stage": round(float(b), 3),
                      "split_share": round(float((nsplit[m] > 1).mean()), 3),
                      "wait_share": round(float(wait[m].sum() / dur[m].sum()), 4)}
    return res


def main(argv=None) -> None:
    import paged_fp8_kv_gk_gb300 as gk
    names = (argv if argv is not None else sys.argv[1:]) or ["gptoss_b64"]
    gk.use_probe_build()
    for name in names:
        print(json.dumps(measure(name)), flush=True)


if __name__ == "__main__":
    main()
