"""DI landing host logic ("GPT-OSS-120B giga-kernel decode", section "DI
wiring (NIXL)"): the region list of a per-layer binding, the block a region's
descriptor lands on, and the N - 1 rule for the sliding-window layers.  Host
only: no device memory is touched (the region calls see plain integers).

Pins: brute-force enumeration of the keys a decode step attends to; the page's
own boundary statement (the at-N window skips a block exactly when
N % block == block - 1); the page's 120B KV-budget byte count for block_len.
"""
import numpy as np
import pytest

import gk_inputs as gi
import oracle
import paged_fp8_kv_gk_gb300 as gk


def _brute(N, B, W):
    """Row blocks of the keys the decode step at position N - 1 reads from the
    transferred cache (keys 0..N-2; the window ones are the last W positions
    up to N - 1 without N - 1 itself)."""
    full = sorted({t // B for t in range(0, N - 1)})
    swa = sorted({t // B for t in range(max(0, N - 1 - W + 1), N - 1)})
    return full, swa


@pytest.mark.parametrize("B", [16, 32, 64, 128])
def test_di_blocks_brute_force_and_oracle(B):
    W = 128
    for N in range(1, 1200):
        full, swa = _brute(N, B, W)
        fc, sf, sc = gk.gk_di_blocks(N, B, W)
        assert fc == len(full) and full == list(range(fc)), (N, B)
        assert sc == len(swa), (N, B)
        if sc:
            assert swa == list(range(sf, sf + sc)), (N, B)
        assert oracle.di_blocks(N, B, W) == (fc, sf, sc)


@pytest.mark.parametrize("B", [16, 32, 64, 128])
def test_at_n_window_drops_a_block_exactly_at_the_page_boundary(B):
    """The page: computing the window at the admitted length N evicts the
    window's oldest block one step early at N % block == block - 1, and that
    block is never transferred.  Brute force over positions: the at-N window
    (keys N - W + 1 .. N - 1) starts a block later than the N - 1 window
    (keys N - W .. N - 2) exactly at that boundary, for N >= W."""
    W = 128
    for N in range(W, 2000):
        at_n = min(t // B for t in range(N - W + 1, N))
        at_n1 = min(t // B for t in range(N - W, N - 1))
        dropped = at_n != at_n1
        assert dropped == (N % B == B - 1), (N, B)
        _, sf, _ = gk.gk_di_blocks(N, B, W)
        assert sf == at_n1
        if dropped:   # the block the fix keeps holds a key the first decode step reads
            assert (N - W) // B == sf


def test_di_blocks_match_the_trimmed_table_and_the_landing_recipe():
    """The decode step at position N - 1 reads its window through a trimmed
    row starting at max(0, N - W) // B: the block gk_di_blocks starts at; the
    landing inputs send exactly gk_di_blocks' counts per row."""
    w = gi.get("di_small")
    c = gi.make_control(w)
    cache = gi.make_cache(w, c)
    dr, db, src = gi.make_landing(w, c, cache)
    B, W = w.block_size, w.window
    per_row = 0
    for b in range(w.batch):
        N = int(c.lengths[b])
        fc, sf, sc = gk.gk_di_blocks(N, B, W)
        assert sf == max(0, N - W) // B
        assert sc <= len(c.swa_blocks[b]) and fc <= len(c.full_blocks[b])
        per_row += fc + sc
    assert dr.size == per_row * 2 * (w.num_layers // 2)
    assert src.shape == (dr.size, w.num_kv_heads * B * w.head_dim)


def test_di_blocks_rejects_bad_arguments():
    for args in [(0, 16, 128), (5, 0, 128), (5, 16, 0)]:
        with pytest.raises(gk.GkError):
            gk.gk_di_blocks(*args)


def _shape(**over):
    d = dict(num_layers=36, batch=1, num_q_heads=64, num_kv_heads=8, head_dim=64, block_size=32,
             num_blocks=1000, window=128, max_blocks_full=8, max_blocks_swa=5)
    d.update(over)
    return gk.Shape.make(**d)


def test_regions_of_the_paired_layer_binding():
    """Layers 2j and 2j+1 bound to group j: 2 * NL/2 regions K_0, V_0, K_1, ...,
    each num_blocks blocks of kv * block * d bytes; the oracle's region list
    (de-duplication by base address) agrees."""
    sh = _shape()
    G = 18
    kb = [0x100000 * (j + 1) for j in range(G)]
    vb = [0x100000 * (j + 1) + 0x80000 for j in range(G)]
    lk = [kb[i // 2] for i in range(36)]
    lv = [vb[i // 2] for i in range(36)]
    r = gk.gk_kv_regions(sh, lk, lv)
    assert len(r) == 2 * G
    assert [x.base for x in r] == [a for j in range(G) for a in (kb[j], vb[j])]
    assert [x.base for x in r] == oracle.kv_regions(lk, lv)
    assert all(x.block_len == 8 * 32 * 64 and x.length == 1000 * 8 * 32 * 64 for x in r)


def test_regions_without_sharing_and_errors():
    sh = _shape(num_layers=4)
    lk = [0x10000 * (i + 1) for i in range(4)]
    lv = [0x10000 * (i + 1) + 0x8000 for i in range(4)]
    r = gk.gk_kv_regions(sh, lk, lv)
    assert [x.base for x in r] == oracle.kv_regions(lk, lv) and len(r) == 8
    with pytest.raises(gk.GkError):
        gk.gk_kv_regions(sh, lk[:3] + [0x10008], lv)      # misaligned
    with pytest.raises(gk.GkError):
        gk.gk_kv_regions(sh, lk[:3] + [0], lv)            # null


def test_block_len_of_the_page_120b_config():
    """The page's 120B GK config: kv_heads 1, block 128, head_size 64, 18 group
    buffers and num_blocks 36,175 come to about 9.94 GiB of KV."""
    sh = _shape(num_layers=36, num_kv_heads=1, block_size=128, num_q_heads=8, num_blocks=36175,
                max_blocks_swa=2)
    lk = [0x1000000 * (i // 2 + 1) for i in range(36)]
    lv = [0x1000000 * (i // 2 + 1) + 0x800000 for i in range(36)]
    r = gk.gk_kv_regions(sh, lk, lv)
    assert r[0].block_len == 8192
    total = sum(x.length for x in r)
    assert abs(total / 2 ** 30 - 9.94) < 0.005


def test_oracle_ingest_is_the_descriptor_definition():
    """Brute-force check of the oracle's landing copy on small arrays: block b
    of region r is bytes [b * block_len, (b + 1) * block_len)."""
    rng = np.random.default_rng(7)
    bl = 32
    regions = [np.zeros(bl * 5, np.uint8) for _ in range(3)]
    pairs = [(0, 4), (2, 0), (1, 1), (2, 3), (7, 0), (0, 9)]   # last two out of range
    src = rng.integers(0, 256, size=(len(pairs), bl), dtype=np.uint8)
    skipped = oracle.kv_ingest(regions, bl, [p[0] for p in pairs], [p[1] for p in pairs], src)
    assert skipped == 2
    want = [np.zeros(bl * 5, np.uint8) for _ in range(3)]
    for d, (r, b) in enumerate(pairs[:4]):
        want[r][b * bl:(b + 1) * bl] = src[d]
    for a, e in zip(regions, want):
        assert np.array_equal(a, e)
