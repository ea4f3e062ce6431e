"""Helpers shared by the GPU parity tests: run one decode step through the C ABI
(via the Python binding), run the oracle on the same inputs, compare.

Tolerances (written here once, used by every parity test):
  * KV bytes after the append: bit-exact.
  * fp32 attention output (out_f32) vs the fp64 oracle: max |d| <= 1.5e-2 and
    mean |d| <= 2e-3.
  * bf16 attention output vs the fp64 oracle: per element
    |d| <= max(1.5e-2, ulp_bf16(oracle)), i.e. the same bar except where one
    bf16 step of the output itself is larger than it (|out| >= 2); and the mean
    of |out - bf16_rne(oracle)| <= 2e-3, the format's own rounding taken out.
"""
from __future__ import annotations

import os

import numpy as np
import torch

import gk_inputs as gi
import oracle
import oracle.rows as oracle_rows
import paged_fp8_kv_gk_gb300 as gk

MAX_ABS = 1.5e-2
MEAN_ABS = 2e-3


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 7), 2.0 ** -133)


# (what, statistics) of every check_out call of the session, listed by the
# terminal summary (tests/conftest.py) so that a quiet run still shows them
REPORT = []


def check_out(out_bf16: np.ndarray, out_f32, ref: np.ndarray, what: str = ""):
    """out_bf16: float64 view of the kernel's bf16 output; out_f32 may be None.
    Returns the error statistics, with `bf16_widened`: how many bf16 elements
    differ from the oracle by more than MAX_ABS and pass only because one bf16
    step of the value is larger than MAX_ABS."""
    d = np.abs(out_bf16 - ref)
    lim = np.maximum(MAX_ABS, ulp_bf16(ref))
    bad = d > lim
    assert not bad.any(), (what, "bf16 max", float(d.max()), np.argwhere(bad)[:5].tolist(),
                           ref[bad][:5].tolist(), out_bf16[bad][:5].tolist())
    mean_r = float(np.mean(np.abs(out_bf16 - oracle.round_bf16(ref)))) if ref.size else 0.0
    assert mean_r <= MEAN_ABS, (what, "bf16 mean", mean_r)
    stats = {"bf16_max": float(d.max()) if d.size else 0.0, "bf16_mean_vs_rne": mean_r,
             "bf16_widened": int(np.count_nonzero(d > MAX_ABS)), "elements": int(d.size)}
    if out_f32 is not None:
        e = np.abs(out_f32 - ref)
        assert e.max() <= MAX_ABS, (what, "f32 max", float(e.max()))
        assert e.mean() <= MEAN_ABS, (what, "f32 mean", float(e.mean()))
        stats.update(f32_max=float(e.max()), f32_mean=float(e.mean()))
    print("check_out", what, {k: (round(v, 6) if isinstance(v, float) else v)
                              for k, v in stats.items()})
    REPORT.append((what, stats))
    return stats


class GpuStep:
    """Inputs of one decode step resident on the GPU, plus the C-ABI calls.

    k_layout: gk.GK_K_PACKED or gk.GK_K_PLAIN (how the K bytes are laid out).
    form: "per_group" (one [2, nb, kv, B, D] buffer per layer pair) or
    "stacked" (K_cache and V_cache with a leading group axis).  Either way
    ``self.cache[j]`` is group j's [2, nb, kv, B, D] (K half, V half)."""

    def __init__(self, w: gi.Workload, c: gi.Control, step: dict, cache, device="cuda",
                 k_layout: int = gk.GK_K_PACKED, form: str = "per_group", sinks=None):
        self.w, self.c = w, c
        dev = torch.device(device)
        self.shape = gk.Shape.make(**gi.shape_dict(w, c))
        t = lambda a, dt: torch.as_tensor(np.ascontiguousarray(a)).to(dev, dt)  # noqa: E731
        self.cos = t(c.cos, torch.float32)
        self.sin = t(c.sin, torch.float32)
        self.k_scale = t(c.k_scale, torch.float32)
        self.v_scale = t(c.v_scale, torch.float32)
        self.bt_full = t(c.bt_full, torch.int32)
        self.bt_swa = t(c.bt_swa, torch.int32)
        self.pos = t(c.pos, torch.int32)
        self.pos_w = t(c.pos_w, torch.int32)
        self.upd_full = t(c.upd_full, torch.int32)
        self.upd_swa = t(c.upd_swa, torch.int32)
        self.active = t(c.active, torch.uint8)
        self.sinks = None if sinks is None else t(sinks, torch.float32)
        self.q = step["q"].to(dev).contiguous()
        self.k_new = step["k_new"].to(dev).contiguous()
        self.v_new = step["v_new"].to(dev).contiguous()
        self.k_layout, self.form = k_layout, form
        if form == "per_group":
            self.cache = [b.to(dev) for b in cache]
            self.kv = gk.kv_from_group_buffers(self.cache, k_layout)
        elif form == "stacked":
            # [2, G, nb, kv, B, D]: K_cache = stack[0], V_cache = stack[1]
            self.stack = torch.stack([torch.stack([b[0] for b in cache]),
                                      torch.stack([b[1] for b in cache])]).to(dev)
            self.cache = [self.stack[:, j] for j in range(len(cache))]
            kc = self.stack[0]
            if k_layout == gk.GK_K_PACKED:
                G, nb, kv, B, D = kc.shape
                kc = kc.view(G, nb, kv, B // 2, D, 2)
            self.kv = gk.kv_stacked(kc, self.stack[1])
        else:
            raise ValueError(form)
        self.out = torch.empty(w.num_layers, w.batch, w.num_q_heads, w.head_dim,
                               dtype=torch.bfloat16, device=dev)
        self.out_f32 = torch.empty(self.out.shape, dtype=torch.float32, device=dev)
        self.workspace = gk.new_workspace(self.shape, dev)

    def append(self, stream=None):
        gk.gk_kv_append(self.shape, self.k_new, self.v_new, self.cos, self.sin, self.k_scale,
                        self.v_scale, self.upd_full, self.upd_swa, self.active, self.kv,
                        stream=stream)

    def step(self, workspace=None, out_f32=True, stream=None):
        """The fused step (gk_decode_step): append + attention in one launch."""
        gk.gk_decode_step(self.shape, self.q, self.k_new, self.v_new, self.cos, self.sin,
                          self.k_scale, self.v_scale, self.upd_full, self.upd_swa, self.bt_full,
                          self.bt_swa, self.pos, self.pos_w, self.active, self.kv,
                          self.out, self.out_f32 if out_f32 else None,
                          self.workspace if workspace is None else workspace, stream=stream,
                          sinks=self.sinks)

    def attention(self, workspace=None, out_f32=True, stream=None):
        gk.gk_decode_attn_stack(self.shape, self.q, self.kv, self.k_scale, self.v_scale,
                                self.cos, self.sin, self.bt_full, self.bt_swa, self.pos,
                                self.pos_w, self.active, self.out,
                                self.out_f32 if out_f32 else None,
                                self.workspace if workspace is None else workspace, stream=stream,
                                sinks=self.sinks)


def oracle_step(w: gi.Workload, c: gi.Control, step: dict, cache, k_layout: int = 0,
                sinks=None):
    """Oracle append + attention on host copies. Returns (out fp64, k_bufs, v_bufs).
    k_layout: 0 packed K view, 1 unpacked K."""
    sh = oracle.make_shape(**gi.shape_dict(w, c), k_layout=k_layout)
    kb = [b[0].cpu().numpy().reshape(-1).copy() for b in cache]
    vb = [b[1].cpu().numpy().reshape(-1).copy() for b in cache]
    st = oracle.kv_append(sh, gi.bf16_bits(step["k_new"]), gi.bf16_bits(step["v_new"]), c.cos,
                          c.sin, c.k_scale, c.v_scale, c.upd_full, c.upd_swa, c.active, kb, vb)
    assert st == 0
    out, st = oracle.decode_attn_stack(sh, gi.bf16_bits(step["q"]), kb, vb, c.k_scale, c.v_scale,
                                       c.cos, c.sin, c.bt_full, c.bt_swa, c.pos, c.pos_w, c.active,
                                       sinks=sinks)
    assert st == 0
    return out, kb, vb


def gather_row_pool(w: gi.Workload, c: gi.Control, cache, j: int, b: int):
    """Host copies of the blocks row b owns in group buffer j (full-layer
    blocks, then window-layer blocks): (K bytes, V bytes)."""
    ids = np.concatenate([np.asarray(c.full_blocks[b], np.int64),
                          np.asarray(c.swa_blocks[b], np.int64)])
    idx = torch.as_tensor(ids, device=cache[j].device)
    return (cache[j][0].index_select(0, idx).cpu().numpy().reshape(-1),
            cache[j][1].index_select(0, idx).cpu().numpy().reshape(-1))


def oracle_row_pair(w: gi.Workload, c: gi.Control, step_host: dict, pre_cache, j: int, b: int,
                    kvhs=None, k_layout: int = 0, sinks=None):
    """Oracle outputs for layers 2j and 2j+1 of row b from the generator's
    pre-append cache (see oracle.rows)."""
    kp, vp = gather_row_pool(w, c, pre_cache, j, b)
    return oracle_rows.row_pair_from_pool(w, c, step_host, kp, vp, j, b, kvhs, k_layout, sinks)


def _k_codes(kbuf, nb, Hkv, B, D, pb, h, t, k_layout):
    """K codes [len(pb), len(h), D] at (pb, h, t) of a K half (numpy or torch)."""
    if k_layout == 0:
        kv = kbuf.reshape(nb, Hkv, B // 2, D, 2)
        return kv[pb[:, None], h[None, :], (t // 2)[:, None], :, (t % 2)[:, None]]
    kv = kbuf.reshape(nb, Hkv, B, D)
    return kv[pb[:, None], h[None, :], t[:, None], :]


def oracle_appended_codes(w: gi.Workload, c: gi.Control, step: dict, k_layout: int = 0):
    """Expected K and V codes of every (layer, row, kv head) the append writes:
    the oracle appends into a compact pool (row b's window layer writes block
    2b, its full layer block 2b+1, at the real in-block offset) and the codes
    are read back from there.  Returns kc, vc [NL, Bt, Hkv, D] uint8."""
    B, Hkv, D, NL, Bt = w.block_size, w.num_kv_heads, w.head_dim, w.num_layers, w.batch
    off = (c.upd_full % B).astype(np.int32)
    assert np.array_equal(off[c.active == 1], (c.upd_swa % B)[c.active == 1])
    upd_s = (2 * np.arange(Bt) * B + off).astype(np.int32)
    upd_f = ((2 * np.arange(Bt) + 1) * B + off).astype(np.int32)
    sh = oracle.make_shape(num_layers=NL, batch=Bt, num_q_heads=w.num_q_heads, num_kv_heads=Hkv,
                           head_dim=D, block_size=B, num_blocks=2 * Bt, window=w.window,
                           max_blocks_full=1, max_blocks_swa=c.max_blocks_swa, k_layout=k_layout)
    nbytes = 2 * Bt * Hkv * B * D
    kb = [np.zeros(nbytes, np.uint8) for _ in range(NL // 2)]
    vb = [np.zeros(nbytes, np.uint8) for _ in range(NL // 2)]
    st = oracle.kv_append(sh, gi.bf16_bits(step["k_new"]), gi.bf16_bits(step["v_new"]), c.cos,
                          c.sin, c.k_scale, c.v_scale, upd_f, upd_s, c.active, kb, vb)
    assert st == 0
    kc = np.zeros((NL, Bt, Hkv, D), np.uint8)
    vc = np.zeros((NL, Bt, Hkv, D), np.uint8)
    for i in range(NL):
        vview = vb[i // 2].reshape(2 * Bt, Hkv, B, D)
        blk = 2 * np.arange(Bt) + (i % 2)
        kc[i] = _k_codes(kb[i // 2], 2 * Bt, Hkv, B, D, blk, np.arange(Hkv), off, k_layout)
        vc[i] = vview[blk[:, None], np.arange(Hkv)[None, :], off[:, None], :]
    return kc, vc


def device_appended_codes(g: GpuStep):
    """Gather the K and V codes at every update slot from the device buffers."""
    w, c = g.w, g.c
    B, Hkv, D, NL, Bt = w.block_size, w.num_kv_heads, w.head_dim, w.num_layers, w.batch
    kc = np.zeros((NL, Bt, Hkv, D), np.uint8)
    vc = np.zeros((NL, Bt, Hkv, D), np.uint8)
    for i in range(NL):
        upd = c.upd_swa if i % 2 == 0 else c.upd_full
        pb = torch.as_tensor((upd // B).astype(np.int64), device=g.cache[0].device)
        t = torch.as_tensor((upd % B).astype(np.int64), device=g.cache[0].device)
        vview = g.cache[i // 2][1]
        hk = torch.arange(Hkv, device=pb.device)
        kc[i] = _k_codes(g.cache[i // 2][0], c.num_blocks, Hkv, B, D, pb, hk, t,
                         g.k_layout).cpu().numpy()
        vc[i] = vview[pb[:, None], hk[None, :], t[:, None], :].cpu().numpy()
    return kc, vc


def host_threads() -> int:
    """Host threads for the oracle: the cores this process may use."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def oracle_full_output(w: gi.Workload, c: gi.Control, step_host: dict, pre_cache,
                       k_layout: int = 0, sinks=None, threads: int = None) -> np.ndarray:
    """The oracle's output for every (layer, row, q head) of a workload of any
    size: [NL, Bt, Hq, D] float64, zero on inactive rows.  Each active row is
    one task (every layer pair, every kv head; oracle.rows.row_all_layers) on
    a pool of host threads (the oracle's C calls release the GIL); a task
    copies its row's blocks from `pre_cache` (the device cache before the
    append) one layer pair at a time.  step_host: q, k_new, v_new as uint16
    bf16 bit arrays."""
    from concurrent.futures import ThreadPoolExecutor
    NL, Bt, Hq, D = w.num_layers, w.batch, w.num_q_heads, w.head_dim
    ref = np.zeros((NL, Bt, Hq, D), np.float64)
    gather = lambda b, j: gather_row_pool(w, c, pre_cache, j, b)  # noqa: E731

    def task(b):
        ref[:, b] = oracle_rows.row_all_layers(w, c, step_host, gather, b, k_layout, sinks)
        return b

    rows = [int(b) for b in np.nonzero(c.active)[0]]
    # longest rows first, so that the pool's last tasks are short ones
    rows.sort(key=lambda b: -int(c.lengths[b]))
    with ThreadPoolExecutor(max_workers=threads or host_threads()) as ex:
        done = list(ex.map(task, rows))
    assert len(done) == len(rows)
    return ref
