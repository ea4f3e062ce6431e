"""Oracle evaluation of single rows of a large workload (test infrastructure).

A full-size workload's cache does not fit the oracle's whole-step call, so one
row at a time is evaluated from a compact pool: the caller copies the blocks
row b owns in group buffer j (its full-layer blocks, then its window-layer
blocks) into host arrays; here they are renumbered, the oracle appends the new
token into them and attends for both layers of the pair.
"""
from __future__ import annotations

import numpy as np

from . import attn_one, kv_append, make_shape


def row_pair_from_pool(w, c, step_host: dict, kpool: np.ndarray, vpool: np.ndarray, j: int,
                       b: int, kvhs=None, k_layout: int = 0, sinks=None) -> dict:
    """w, c: the workload and its control tensors (gk_inputs.Workload/Control).
    step_host: q, k_new, v_new as uint16 bf16 bit arrays.  kpool/vpool: bytes
    of row b's full blocks followed by its window blocks (K halves and V
    halves, each block Hkv*B*D bytes), from the cache before the append.
    k_layout: 0 packed K view, 1 unpacked K.  sinks: optional [NL, Hq] sink logits.
    Returns {(layer, kvh): [G, D] float64} for layers 2j and 2j+1."""
    B, Hkv, D, NL = w.block_size, w.num_kv_heads, w.head_dim, w.num_layers
    kvhs = range(Hkv) if kvhs is None else kvhs
    nf, ns_ = len(c.full_blocks[b]), len(c.swa_blocks[b])
    per_blk = Hkv * B * D
    assert kpool.size == (nf + ns_) * per_blk and vpool.size == kpool.size
    kmini = np.concatenate([kpool.reshape(-1), np.zeros(per_blk, np.uint8)])
    vmini = np.concatenate([vpool.reshape(-1), np.zeros(per_blk, np.uint8)])
    pad = nf + ns_
    mbf = max(1, nf)
    bt_full = np.full((1, mbf), pad, np.int32)
    bt_full[0, :nf] = np.arange(nf)
    bt_swa = np.full((1, c.max_blocks_swa), pad, np.int32)
    bt_swa[0, :ns_] = nf + np.arange(ns_)
    pos = int(c.pos[b])
    upd_f = np.array([bt_full[0, pos // B] * B + pos % B], np.int32)
    b0 = (pos - int(c.pos_w[b])) // B
    upd_s = np.array([bt_swa[0, pos // B - b0] * B + pos % B], np.int32)
    sh = make_shape(num_layers=NL, batch=1, num_q_heads=w.num_q_heads, num_kv_heads=Hkv,
                    head_dim=D, block_size=B, num_blocks=pad + 1, window=w.window,
                    max_blocks_full=mbf, max_blocks_swa=c.max_blocks_swa, k_layout=k_layout)
    # only group j's pool is real; the other groups get scratch pools
    scratch_k = [np.zeros(kmini.size, np.uint8) for _ in range(NL // 2)]
    scratch_v = [np.zeros(vmini.size, np.uint8) for _ in range(NL // 2)]
    scratch_k[j], scratch_v[j] = kmini, vmini
    row = lambda a: np.ascontiguousarray(a[:, b:b + 1])  # noqa: E731
    st = kv_append(sh, row(step_host["k_new"]), row(step_host["v_new"]), c.cos[b:b + 1],
                   c.sin[b:b + 1], c.k_scale, c.v_scale, upd_f, upd_s, c.active[b:b + 1],
                   scratch_k, scratch_v)
    assert st == 0
    res = {}
    for layer in (2 * j, 2 * j + 1):
        for kvh in kvhs:
            out, st = attn_one(sh, row(step_host["q"]), kmini, vmini, c.k_scale, c.v_scale,
                               c.cos[b:b + 1], c.sin[b:b + 1], bt_full, bt_swa, c.pos[b:b + 1],
                               c.pos_w[b:b + 1], c.active[b:b + 1], layer, 0, kvh, sinks=sinks)
            assert st == 0
            res[(layer, kvh)] = out
    return res


def row_all_layers(w, c, step_host: dict, gather, b: int, k_layout: int = 0,
                   sinks=None) -> np.ndarray:
    """Oracle output of row b for every layer and q head: [NL, Hq, D] float64.
    gather(b, j) returns the (K pool, V pool) of row b in group buffer j as
    row_pair_from_pool expects them (from the cache before the append); it is
    called once per layer pair, so that only one pair's pools are held at a
    time."""
    NL, Hq, D, Hkv = w.num_layers, w.num_q_heads, w.head_dim, w.num_kv_heads
    G = Hq // Hkv
    out = np.zeros((NL, Hq, D), np.float64)
    for j in range(NL // 2):
        kp, vp = gather(b, j)
        res = row_pair_from_pool(w, c, step_host, kp, vp, j, b, None, k_layout, sinks)
        for (layer, kvh), o in res.items():
            out[layer, kvh * G:(kvh + 1) * G] = o
    return out
