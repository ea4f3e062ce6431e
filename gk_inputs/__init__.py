"""Seeded synthetic workloads for the stack-wide paged-FP8 decode-attention step.

This module only draws inputs: shapes, context lengths, block tables, the
attention-control tensors a caller builds for one decode step, random q/k/v and
a pre-filled KV cache.  It holds none of the step's arithmetic (no RoPE, no
attention, no quantiser of its own) and is shared by both sides of the parity
tests: the oracle and the CUDA library each consume what it produces.

Control tensors follow "GPT-OSS-120B giga-kernel decode", section "Kernel
contract": RoPE cos/sin, a full block table and a trimmed sliding-window block
table, an active mask, absolute and window-frame positions, and the two KV
update indices.  Blocks come from one pool per group buffer with disjoint ids
for the sliding-window and the full layer that share it (section "KV-cache
layout").  The last block of the pool is a padding block that no table row
references except as padding.

Workload recipe (stated once, used everywhere):
  * context length L_b counts the new token; its position is pos_b = L_b - 1;
  * the full layer of sequence b owns ceil(L_b / B) blocks, the sliding-window
    layer owns the blocks b0 .. pos_b // B with b0 = max(0, L_b - W) // B; the
    trimmed row starts at b0, the window-frame position is pos_w = pos_b - b0*B;
  * update index = physical block * B + offset of pos_b in its block (full and
    trimmed row respectively); inactive rows point at the padding block;
  * physical block ids are one random permutation of [0, nb - 1) handed out in
    sequence order; nb = blocks used + 1 unless the workload fixes it;
  * cos/sin rows: angle pos_b * theta^(-2e/D), e < D/2, in double, stored fp32;
  * q ~ N(0, sigma_q), k_new and v_new ~ N(0, sigma), drawn in fp32 and
    rounded to bf16 (the short-context workload's "KV values ~ N(0, 3)" is read
    as sigma = 3 for K and V only; q stays N(0, 1));
  * cache bytes: codes of N(0, sigma_cache) / scale, drawn by torch and cast
    with torch's float8_e4m3fn conversion after clamping to +-448 (a library
    cast; the cache is an input like any other);
  * the saturation probe sets a seeded 1/1024 of k_new/v_new to +-U(28, 60).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np
import torch

E4M3_MAX = 448.0


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    num_layers: int
    batch: int
    num_q_heads: int
    num_kv_heads: int
    block_size: int
    lengths: str                  # "fixed:a,b,.." | "uniform:lo,hi" | "loguniform:lo,hi" | "all:n"
    seed: int
    head_dim: int = 64
    window: int = 128
    inactive_frac: float = 0.0
    sigma: float = 1.0            # k_new, v_new
    sigma_q: float = 1.0          # q
    sigma_cache: float = 1.0      # pre-filled cache values (before 1/scale)
    scale: Optional[float] = None  # None: per-layer 2^-(4 + i mod 3)
    theta: float = 150000.0
    num_blocks: Optional[int] = None
    sat_probe: bool = False
    description: str = ""

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads of the decode-attention measurement, plus the saturation
# probe variant of the short-context one.
WORKLOADS = {
    "tiny": Workload("tiny", 2, 2, 8, 1, 16, "fixed:40,200", seed=0, scale=1 / 64, num_blocks=64,
                     description="2 layers (SWA-128 + full) sharing one buffer, batch 2, L 40 and 200, "
                                 "8 q / 1 kv heads, block 16, 64 blocks, scale 1/64"),
    "gptoss_b64": Workload("gptoss_b64", 36, 64, 64, 8, 32, "uniform:1024,8192", seed=2,
                           description="GPT-OSS-120B attention shapes: 36 layers, batch 64, "
                                       "64 q / 8 kv heads, block 32, L ~ U{1024..8192}"),
    "long_ctx": Workload("long_ctx", 36, 8, 64, 8, 32, "all:131072", seed=3,
                         description="36 layers, batch 8, every context 131072 tokens"),
    "ragged_b256": Workload("ragged_b256", 36, 256, 64, 8, 32, "loguniform:128,32768", seed=4,
                            inactive_frac=0.10,
                            description="36 layers, batch 256, L log-uniform [128, 32768], "
                                        "10% of rows inactive"),
    "swa_b512": Workload("swa_b512", 36, 512, 64, 8, 32, "uniform:64,512", seed=5, sigma=3.0,
                         sigma_cache=3.0, scale=1 / 16,
                         description="36 layers, batch 512, L ~ U{64..512}, KV values N(0, 3), "
                                     "q N(0, 1), scale 1/16"),
}
WORKLOADS["swa_b512_sat"] = WORKLOADS["swa_b512"].replace(
    name="swa_b512_sat", sat_probe=True,
    description="swa_b512 with a seeded 1/1024 of new K/V set to +-U(28, 60) (saturates at 448)")

# Reduced versions the oracle finishes in seconds: same structure, fewer
# layers/rows, lengths chosen to hit block-boundary and window-boundary cases.
REDUCED = {
    "gptoss_small": WORKLOADS["gptoss_b64"].replace(
        name="gptoss_small", num_layers=4, batch=6, lengths="fixed:1,31,32,159,160,1100", seed=12),
    "long_small": WORKLOADS["long_ctx"].replace(
        name="long_small", num_layers=2, batch=2, lengths="all:9000", seed=13),
    # three rows long enough that equal chunks leave a partial last wave, so
    # the planner cuts chunks of the long rows into pieces for it (checked on
    # sampled rows: the whole-step oracle would take about a minute)
    "long_cut_small": WORKLOADS["long_ctx"].replace(
        name="long_cut_small", num_layers=16, batch=3, lengths="all:36000", seed=32),
    "ragged_small": WORKLOADS["ragged_b256"].replace(
        name="ragged_small", num_layers=4, batch=12, lengths="loguniform:1,3000", seed=14,
        inactive_frac=0.25),
    "swa_small": WORKLOADS["swa_b512"].replace(
        name="swa_small", num_layers=4, batch=16, lengths="uniform:64,512", seed=15),
    "swa_small_sat": WORKLOADS["swa_b512_sat"].replace(
        name="swa_small_sat", num_layers=4, batch=16, lengths="uniform:64,512", seed=16),
    # stress variant, not one of the five workloads: q ~ N(0, 3) as well, so
    # logits have a standard deviation near 9 and the softmax is very peaked
    "swa_small_peaky": WORKLOADS["swa_b512"].replace(
        name="swa_small_peaky", num_layers=4, batch=16, lengths="uniform:64,512", seed=18,
        sigma_q=3.0),
    # block 128 with one kv head: the page's 120B GK config seen by one TP8 rank
    "gk120b_rank_small": WORKLOADS["tiny"].replace(
        name="gk120b_rank_small", num_layers=4, batch=5, block_size=128,
        lengths="fixed:1,127,128,129,700", seed=19, num_blocks=None, scale=None),
    "block64_small": WORKLOADS["gptoss_b64"].replace(
        name="block64_small", num_layers=4, batch=5, block_size=64,
        lengths="fixed:1,63,64,200,1000", seed=20),
    "block16_small": WORKLOADS["tiny"].replace(
        name="block16_small", num_layers=4, batch=5, num_q_heads=16, num_kv_heads=2,
        lengths="fixed:1,15,16,143,300", seed=17, num_blocks=None),
    # the largest shapes the library accepts: batch 8192, 1024-token blocks,
    # 128 layers (64 group buffers)
    "max_batch": WORKLOADS["tiny"].replace(
        name="max_batch", batch=8192, lengths="uniform:1,64", seed=27, num_blocks=None),
    "max_block": WORKLOADS["tiny"].replace(
        name="max_block", num_layers=4, batch=3, block_size=1024, lengths="fixed:1,1000,2500",
        seed=28, num_blocks=None),
    "max_layers": WORKLOADS["tiny"].replace(
        name="max_layers", num_layers=128, batch=2, block_size=32, lengths="fixed:40,300",
        seed=29, num_blocks=None, scale=None),
    # forced split lengths: at 512-token chunks these rows take 1, 2, 7 and
    # 64 chunks (the cap per row; the last row's final chunk holds one key)
    "split_counts_small": WORKLOADS["gptoss_b64"].replace(
        name="split_counts_small", num_layers=4, batch=5, lengths="fixed:300,1000,3500,32768,32257",
        seed=33),
    # DI landing: prompt lengths on both sides of N % B == B - 1 (143, 159 with
    # N >= W; 127 below it), a one-token prompt and block-boundary lengths
    "di_small": WORKLOADS["gptoss_b64"].replace(
        name="di_small", num_layers=4, batch=8, block_size=16,
        lengths="fixed:1,2,127,128,143,159,160,700", seed=25),
}

# KV landing measurement: 16 prompts of 8192 tokens at the 36-layer shapes
# (about 2.4 GB of blocks landed per step).
LANDING = {
    "di_ingest_b16": WORKLOADS["gptoss_b64"].replace(
        name="di_ingest_b16", batch=16, lengths="all:8192", seed=26),
}


# Profiling size of the 36-layer workload: same per-row shape, 8 rows, about
# 0.7 GB of KV per step (larger than L2, small enough for a full counter set).
PROFILE = {
    "gptoss_b8": WORKLOADS["gptoss_b64"].replace(name="gptoss_b8", batch=8, seed=22),
    "gptoss_b16": WORKLOADS["gptoss_b64"].replace(name="gptoss_b16", batch=16, seed=23),
    "swa_b128": WORKLOADS["swa_b512"].replace(name="swa_b128", batch=128, seed=24),
    # latency end of the 36-layer shapes: one or eight rows of 8192 tokens
    # (0.15 / 1.2 GB of KV), where the fixed costs of a call weigh most
    "gptoss_b1_8k": WORKLOADS["gptoss_b64"].replace(name="gptoss_b1_8k", batch=1,
                                                     lengths="all:8192", seed=30),
    "gptoss_b8_8k": WORKLOADS["gptoss_b64"].replace(name="gptoss_b8_8k", batch=8,
                                                     lengths="all:8192", seed=31),
    # reduced cases of the long-context and ragged workloads (a few GB of KV)
    # for DRAM counters, scaled to the full workloads by algorithmic bytes
    "long_b1": WORKLOADS["long_ctx"].replace(name="long_b1", batch=1, seed=35),
    "ragged_b24": WORKLOADS["ragged_b256"].replace(name="ragged_b24", batch=24, seed=36),
}

# The page's deployed per-rank shape of the 120B GK decode (TP8: one kv head
# per rank, 8 q heads, block 128, head 64) over the 36-layer stack, with the
# batch and context mix of the batch-64 workload.
RANK = {
    "gk120b_rank_b64": WORKLOADS["gptoss_b64"].replace(
        name="gk120b_rank_b64", num_q_heads=8, num_kv_heads=1, block_size=128, seed=37,
        description="36 layers, batch 64, 8 q / 1 kv heads (one TP8 rank), block 128, "
                    "L ~ U{1024..8192}"),
}


def get(name: str) -> Workload:
    for table in (WORKLOADS, REDUCED, PROFILE, LANDING, RANK):
        if name in table:
            return table[name]
    raise KeyError(name)


@dataclasses.dataclass
class Control:
    """Layer-invariant control tensors of one decode step (numpy, host)."""
    lengths: np.ndarray     # int64 [Bt]  (0 for inactive rows)
    active: np.ndarray      # uint8 [Bt]
    pos: np.ndarray         # int32 [Bt]
    pos_w: np.ndarray       # int32 [Bt]
    bt_full: np.ndarray     # int32 [Bt, MBF]
    bt_swa: np.ndarray      # int32 [Bt, MBS]
    upd_full: np.ndarray    # int32 [Bt]
    upd_swa: np.ndarray     # int32 [Bt]
    cos: np.ndarray         # float32 [Bt, D/2]
    sin: np.ndarray         # float32 [Bt, D/2]
    k_scale: np.ndarray     # float32 [NL]
    v_scale: np.ndarray     # float32 [NL]
    num_blocks: int
    max_blocks_full: int
    max_blocks_swa: int
    full_blocks: List[np.ndarray]   # physical ids per row, full layer
    swa_blocks: List[np.ndarray]    # physical ids per row, sliding-window layer (from b0)

    @property
    def padding_block(self) -> int:
        return self.num_blocks - 1


def _lengths(w: Workload, rng: np.random.Generator) -> np.ndarray:
    kind, _, arg = w.lengths.partition(":")
    if kind == "fixed":
        vals = [int(x) for x in arg.split(",")]
        assert len(vals) == w.batch
        return np.array(vals, np.int64)
    if kind == "all":
        return np.full(w.batch, int(arg), np.int64)
    lo, hi = (int(x) for x in arg.split(","))
    if kind == "uniform":
        return rng.integers(lo, hi + 1, size=w.batch).astype(np.int64)
    if kind == "loguniform":
        u = rng.uniform(math.log(lo), math.log(hi), size=w.batch)
        return np.clip(np.round(np.exp(u)), lo, hi).astype(np.int64)
    raise ValueError(w.lengths)


def layer_scales(w: Workload) -> np.ndarray:
    if w.scale is not None:
        return np.full(w.num_layers, w.scale, np.float32)
    return np.array([2.0 ** -(4 + (i % 3)) for i in range(w.num_layers)], np.float32)


def make_control(w: Workload) -> Control:
    rng = np.random.default_rng(w.seed)
    B, W, D = w.block_size, w.window, w.head_dim
    L = _lengths(w, rng)
    active = np.ones(w.batch, np.uint8)
    if w.inactive_frac > 0:
        n_in = int(round(w.inactive_frac * w.batch))
        active[rng.choice(w.batch, size=n_in, replace=False)] = 0
    L = np.where(active == 1, L, 0)

    n_full = [(-(-int(l) // B)) if a else 0 for l, a in zip(L, active)]
    b0 = [max(0, int(l) - W) // B for l in L]
    n_swa = [((int(l) - 1) // B - s + 1) if a else 0 for l, a, s in zip(L, active, b0)]
    used = sum(n_full) + sum(n_swa)
    nb = w.num_blocks if w.num_blocks is not None else used + 1
    if used + 1 > nb:
        raise ValueError(f"{w.name}: needs {used + 1} blocks, pool has {nb}")
    perm = rng.permutation(nb - 1).astype(np.int64)
    mbf = max(1, max(n_full))
    mbs = -(-(W + B - 1) // B)
    pad = nb - 1
    bt_full = np.full((w.batch, mbf), pad, np.int32)
    bt_swa = np.full((w.batch, mbs), pad, np.int32)
    full_blocks, swa_blocks = [], []
    cur = 0
    for b in range(w.batch):
        fb = perm[cur:cur + n_full[b]]
        cur += n_full[b]
        sb = perm[cur:cur + n_swa[b]]
        cur += n_swa[b]
        bt_full[b, :len(fb)] = fb
        bt_swa[b, :len(sb)] = sb
        full_blocks.append(fb)
        swa_blocks.append(sb)

    pos = np.where(active == 1, L - 1, 0).astype(np.int32)
    pos_w = np.array([(p - s * B) if a else 0 for p, s, a in zip(pos, b0, active)], np.int32)
    upd_full = np.full(w.batch, pad * B, np.int32)
    upd_swa = np.full(w.batch, pad * B, np.int32)
    for b in range(w.batch):
        if active[b]:
            p = int(pos[b])
            upd_full[b] = int(bt_full[b, p // B]) * B + p % B
            upd_swa[b] = int(bt_swa[b, p // B - b0[b]]) * B + p % B

    inv = w.theta ** (-(2.0 * np.arange(D // 2, dtype=np.float64)) / D)
    ang = pos.astype(np.float64)[:, None] * inv[None, :]
    sc = layer_scales(w)
    return Control(lengths=L, active=active, pos=pos, pos_w=pos_w, bt_full=bt_full, bt_swa=bt_swa,
                   upd_full=upd_full, upd_swa=upd_swa, cos=np.cos(ang).astype(np.float32),
                   sin=np.sin(ang).astype(np.float32), k_scale=sc.copy(), v_scale=sc.copy(),
                   num_blocks=nb, max_blocks_full=mbf, max_blocks_swa=mbs,
                   full_blocks=full_blocks, swa_blocks=swa_blocks)


def shape_dict(w: Workload, c: Control) -> dict:
    return dict(num_layers=w.num_layers, batch=w.batch, num_q_heads=w.num_q_heads,
                num_kv_heads=w.num_kv_heads, head_dim=w.head_dim, block_size=w.block_size,
                num_blocks=c.num_blocks, window=w.window, max_blocks_full=c.max_blocks_full,
                max_blocks_swa=c.max_blocks_swa)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_step(w: Workload, device="cpu") -> dict:
    """q [NL,Bt,Hq,D], k_new and v_new [NL,Bt,Hkv,D]: bf16 torch tensors."""
    g = _gen(device, w.seed * 7919 + 1)
    NL, Bt, D = w.num_layers, w.batch, w.head_dim
    q = (torch.randn(NL, Bt, w.num_q_heads, D, generator=g, device=device) * w.sigma_q).to(torch.bfloat16)
    k = (torch.randn(NL, Bt, w.num_kv_heads, D, generator=g, device=device) * w.sigma)
    v = (torch.randn(NL, Bt, w.num_kv_heads, D, generator=g, device=device) * w.sigma)
    if w.sat_probe:
        for t in (k, v):
            n = t.numel()
            m = max(1, n // 1024)
            idx = torch.randperm(n, generator=g, device=device)[:m]
            mag = torch.rand(m, generator=g, device=device) * 32.0 + 28.0
            sgn = torch.where(torch.rand(m, generator=g, device=device) < 0.5, -1.0, 1.0)
            t.view(-1)[idx] = mag * sgn
    return dict(q=q, k_new=k.to(torch.bfloat16), v_new=v.to(torch.bfloat16))


def _codes(n: int, sigma_over_scale: float, g: torch.Generator, device) -> torch.Tensor:
    x = torch.randn(n, generator=g, device=device) * sigma_over_scale
    return x.clamp_(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8)


def make_cache(w: Workload, c: Control, device="cpu", chunk: int = 1 << 27) -> List[torch.Tensor]:
    """One uint8 tensor [2, nb, Hkv, B, D] per group buffer (K half, then V half).
    Every block gets codes drawn at the full layer's scale; the blocks the
    sliding-window layer owns are then redrawn at that layer's scale."""
    g = _gen(device, w.seed * 104729 + 3)
    per_blk = w.num_kv_heads * w.block_size * w.head_dim
    swa_ids = np.concatenate([s for s in c.swa_blocks if len(s)] or [np.zeros(0, np.int64)])
    swa_ids_t = torch.as_tensor(swa_ids, dtype=torch.long, device=device)
    bufs = []
    for j in range(w.num_layers // 2):
        buf = torch.empty(2, c.num_blocks, w.num_kv_heads, w.block_size, w.head_dim,
                          dtype=torch.uint8, device=device)
        flat = buf.view(-1)
        s_full = w.sigma_cache / float(c.k_scale[2 * j + 1])
        for o in range(0, flat.numel(), chunk):
            n = min(chunk, flat.numel() - o)
            flat[o:o + n] = _codes(n, s_full, g, device)
        if swa_ids_t.numel():
            s_swa = w.sigma_cache / float(c.k_scale[2 * j])
            for half in range(2):
                blk = buf[half].view(c.num_blocks, per_blk)
                blk[swa_ids_t] = _codes(swa_ids_t.numel() * per_blk, s_swa, g, device).view(-1, per_blk)
        bufs.append(buf)
    return bufs


def make_landing(w: Workload, c: Control, cache: List[torch.Tensor]):
    """DI landing inputs ("GPT-OSS-120B giga-kernel decode", section "DI wiring
    (NIXL)"): the blocks a prefill engine sends for every active row b, a
    prompt of N = L_b tokens whose last token the decode engine recomputes at
    position N - 1 (both engines operate at N - 1), so keys 0 .. N-2:
      * full layer: row blocks 0 .. ceil((N-1)/B) - 1 (entries of bt_full);
      * window layer: the trimmed row's entries for keys max(0, N-W) .. N-2
        (the row starts at block max(0, N-W) // B).
    Regions: 2j = group j's K half, 2j + 1 its V half.  Returns
    (dst_region int32 [n], dst_block int32 [n], src uint8 [n, block_len]) with
    src taken from `cache` (the bytes the prefill engine holds), on its device."""
    B, W = w.block_size, w.window
    regs, blks = [], []
    for b in range(w.batch):
        if not c.active[b]:
            continue
        N = int(c.lengths[b])
        nf = -(-(N - 1) // B)
        lo = max(0, N - W)
        ns = (N - 2) // B - lo // B + 1 if N - 2 >= lo else 0
        ids = [int(x) for x in c.full_blocks[b][:nf]] + [int(x) for x in c.swa_blocks[b][:ns]]
        for j in range(w.num_layers // 2):
            for half in range(2):
                regs += [2 * j + half] * len(ids)
                blks += ids
    dst_region = np.asarray(regs, np.int32)
    dst_block = np.asarray(blks, np.int32)
    per_blk = w.num_kv_heads * B * w.head_dim
    dev = cache[0].device
    src = torch.empty(len(regs), per_blk, dtype=torch.uint8, device=dev)
    r_t = torch.as_tensor(dst_region, device=dev, dtype=torch.long)
    b_t = torch.as_tensor(dst_block, device=dev, dtype=torch.long)
    for r in range(2 * (w.num_layers // 2)):
        sel = (r_t == r).nonzero().view(-1)
        if sel.numel():
            src[sel] = cache[r // 2][r % 2].view(c.num_blocks, per_blk).index_select(0, b_t[sel])
    return dst_region, dst_block, src


def make_sinks(w: Workload, seed: int = 0) -> np.ndarray:
    """Attention-sink logits fp32 [NL, Hq] (natural-log units, the scale of the
    scores): N(0, 2), with every 7th head set to +12 (the sink dominates the
    row) and every 11th to -30 (it vanishes)."""
    rng = np.random.default_rng(w.seed * 7919 + 11 + seed)
    s = rng.normal(0.0, 2.0, (w.num_layers, w.num_q_heads))
    h = np.arange(w.num_q_heads)
    s[:, h % 7 == 3] = 12.0
    s[:, h % 11 == 5] = -30.0
    return s.astype(np.float32)


def kv_bytes_read(w: Workload, c: Control) -> int:
    """Algorithmic KV bytes one decode-attention step reads: each active row
    reads Hkv * D bytes of K and of V per key, L keys in full layers and
    min(L, W) keys in sliding-window layers."""
    per_key = w.num_kv_heads * w.head_dim * 2
    n_full = int(sum(int(l) for l, a in zip(c.lengths, c.active) if a))
    n_swa = int(sum(min(int(l), w.window) for l, a in zip(c.lengths, c.active) if a))
    half = w.num_layers // 2
    return per_key * half * (n_full + n_swa)


def qo_bytes(w: Workload, c: Control) -> int:
    """Algorithmic q read + out write bytes (bf16) for the active rows."""
    n_act = int(c.active.sum())
    return 2 * w.num_layers * n_act * w.num_q_heads * w.head_dim * 2


def layer_seqs(w: Workload, c: Control) -> int:
    return w.num_layers * int(c.active.sum())


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 torch tensor -> numpy uint16 bit patterns (host)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
