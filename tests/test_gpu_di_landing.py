"""GPU parity of the DI landing copy (gk_kv_ingest; "GPT-OSS-120B giga-kernel
decode", section "DI wiring (NIXL)"): every landed byte bit-exact against the
oracle's copy by the descriptor definition; out-of-range descriptors skipped
with the device error bit; a pinned host source; the stacked KV form; and the
landing followed by a decode step, which must give the outputs of the step on
the prefill engine's own cache, and which differs when the window blocks are
chosen by the at-N rule the page replaced.
"""
import numpy as np
import pytest
import torch

import gk_inputs as gi
import gk_testlib as tl
import oracle
import paged_fp8_kv_gk_gb300 as gk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    gk.lib()
    gk.gk_read_device_error(clear=True)
    yield
    torch.cuda.synchronize()


def _fresh_cache(w, c, dev="cuda"):
    return [torch.zeros(2, c.num_blocks, w.num_kv_heads, w.block_size, w.head_dim,
                        dtype=torch.uint8, device=dev) for _ in range(w.num_layers // 2)]


def _regions(w, c, kv):
    lk, lv = gk.layer_binding(kv, w.num_layers)
    return gk.gk_kv_regions(gk.Shape.make(**gi.shape_dict(w, c)), lk, lv)


def _oracle_land(w, c, dst_region, dst_block, src):
    per_blk = w.num_kv_heads * w.block_size * w.head_dim
    regs = [np.zeros(c.num_blocks * per_blk, np.uint8) for _ in range(w.num_layers)]
    skipped = oracle.kv_ingest(regs, per_blk, dst_region, dst_block, src.cpu().numpy())
    return regs, skipped


def _device_regions(cache):
    return [h.reshape(-1).cpu().numpy() for b in cache for h in (b[0], b[1])]


@pytest.mark.parametrize("form", ["per_group", "stacked"])
def test_landing_bytes_exact(form):
    w = gi.get("di_small")
    c = gi.make_control(w)
    truth = gi.make_cache(w, c, "cuda")
    dr, db, src = gi.make_landing(w, c, truth)
    cache = _fresh_cache(w, c)
    if form == "stacked":
        kst = torch.stack([b[0] for b in cache])
        vst = torch.stack([b[1] for b in cache])
        kv = gk.kv_stacked(kst, vst)
        views = [torch.stack((kst[j], vst[j])) for j in range(len(cache))]
    else:
        kv = gk.kv_from_group_buffers(cache, gk.GK_K_PLAIN)
    regions = _regions(w, c, kv)
    assert len(regions) == w.num_layers
    gk.gk_kv_ingest(regions, torch.as_tensor(dr, device="cuda"),
                    torch.as_tensor(db, device="cuda"), src)
    torch.cuda.synchronize()
    assert gk.gk_read_device_error() == 0
    if form == "stacked":
        cache = [torch.stack((kst[j], vst[j])) for j in range(len(cache))]
    want, skipped = _oracle_land(w, c, dr, db, src)
    assert skipped == 0
    for r, (a, e) in enumerate(zip(_device_regions(cache), want)):
        assert np.array_equal(a, e), r


def test_out_of_range_descriptors_skipped_and_flagged():
    w = gi.get("di_small")
    c = gi.make_control(w)
    truth = gi.make_cache(w, c, "cuda")
    dr, db, src = gi.make_landing(w, c, truth)
    dr = dr.copy()
    db = db.copy()
    dr[3] = w.num_layers          # region past the list
    db[7] = c.num_blocks          # block past the region
    db[9] = -1
    cache = _fresh_cache(w, c)
    kv = gk.kv_from_group_buffers(cache)
    gk.gk_kv_ingest(_regions(w, c, kv), torch.as_tensor(dr, device="cuda"),
                    torch.as_tensor(db, device="cuda"), src)
    assert gk.gk_read_device_error() == gk.GK_DEVERR_INGEST
    want, skipped = _oracle_land(w, c, dr, db, src)
    assert skipped == 3
    for a, e in zip(_device_regions(cache), want):
        assert np.array_equal(a, e)


def test_pinned_host_source():
    w = gi.get("di_small")
    c = gi.make_control(w)
    truth = gi.make_cache(w, c, "cuda")
    dr, db, src = gi.make_landing(w, c, truth)
    host = src.cpu().pin_memory()
    cache = _fresh_cache(w, c)
    kv = gk.kv_from_group_buffers(cache)
    gk.gk_kv_ingest(_regions(w, c, kv), torch.as_tensor(dr, device="cuda"),
                    torch.as_tensor(db, device="cuda"), host)
    torch.cuda.synchronize()
    assert gk.gk_read_device_error() == 0
    want, _ = _oracle_land(w, c, dr, db, src)
    for a, e in zip(_device_regions(cache), want):
        assert np.array_equal(a, e)


def test_pageable_host_source_refused():
    w = gi.get("di_small")
    c = gi.make_control(w)
    cache = _fresh_cache(w, c)
    kv = gk.kv_from_group_buffers(cache)
    regions = _regions(w, c, kv)
    src = torch.zeros(2, w.num_kv_heads * w.block_size * w.head_dim, dtype=torch.uint8)
    idx = torch.zeros(2, dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        gk.gk_kv_ingest(regions, idx, idx, src)
    # the library itself refuses it too (the binding's check bypassed): plain
    # pageable memory is not an address the kernel may read
    arr = np.zeros(2 * w.num_kv_heads * w.block_size * w.head_dim + 16, np.uint8)
    addr = (arr.ctypes.data + 15) // 16 * 16
    st = gk.lib().gk_kv_ingest(regions, len(regions), idx.data_ptr(), idx.data_ptr(), 2, addr,
                               None)
    assert st == gk.GK_ERR_INVALID_ARG


def _landed_step(w, c, st, truth, swa_rule="n_minus_1"):
    """Land the prefill engine's blocks on a fresh decode cache, then run the
    decode step (append + attention) there."""
    dr, db, src = gi.make_landing(w, c, truth)
    if swa_rule == "at_n":
        # the rule the page replaced: the window computed for length N keeps
        # keys from N - W + 1, so at N % B == B - 1 (N >= W) the first block
        # of the trimmed row is not sent
        keep = np.ones(dr.size, bool)
        B, W = w.block_size, w.window
        for b in range(w.batch):
            N = int(c.lengths[b])
            if c.active[b] and N >= W and N % B == B - 1:
                keep &= db != int(c.swa_blocks[b][0])
        dr, db, src = dr[keep], db[keep], src[torch.as_tensor(keep, device=src.device)]
    cache = _fresh_cache(w, c)
    g = tl.GpuStep(w, c, st, cache)
    gk.gk_kv_ingest(_regions(w, c, g.kv), torch.as_tensor(dr, device="cuda"),
                    torch.as_tensor(db, device="cuda"), src)
    g.append()
    g.attention()
    torch.cuda.synchronize()
    return g


def test_landing_then_decode_matches_the_prefill_cache():
    w = gi.get("di_small")
    c = gi.make_control(w)
    st = gi.make_step(w, "cpu")
    truth = gi.make_cache(w, c, "cuda")
    ref = tl.GpuStep(w, c, st, [b.clone() for b in truth])
    ref.append()
    ref.attention()
    got = _landed_step(w, c, st, truth)
    assert gk.gk_read_device_error() == 0
    # keys outside the landed blocks are masked, so the outputs are bit-identical
    assert torch.equal(got.out, ref.out) and torch.equal(got.out_f32, ref.out_f32)
    # and they are the oracle's within the parity tolerance
    cpu = [b.cpu() for b in truth]
    want, _, _ = tl.oracle_step(w, c, st, cpu)
    tl.check_out(got.out.float().cpu().numpy().astype(np.float64),
                 got.out_f32.cpu().numpy().astype(np.float64), want, "landed step")


def test_at_n_rule_loses_the_boundary_block():
    w = gi.get("di_small")
    c = gi.make_control(w)
    st = gi.make_step(w, "cpu")
    truth = gi.make_cache(w, c, "cuda")
    good = _landed_step(w, c, st, truth)
    bad = _landed_step(w, c, st, truth, swa_rule="at_n")
    B, W = w.block_size, w.window
    hit = [b for b in range(w.batch)
           if c.active[b] and int(c.lengths[b]) >= W and int(c.lengths[b]) % B == B - 1]
    assert hit, "the workload must contain a boundary row"
    swa_layers = list(range(0, w.num_layers, 2))
    for b in range(w.batch):
        same = torch.equal(good.out_f32[swa_layers, b], bad.out_f32[swa_layers, b])
        assert same == (b not in hit), b
