"""Oracle pins for the unpacked-K layout ("GPT-OSS-120B giga-kernel decode",
section "KV-cache layout": the packed K is a trailing view of the same bytes,
``[.., block // 2, d, 2]``; the unpacked K is ``[.., block, d]`` like V, and the
kernel reads which one it has from the K rank).

The unpacked layout is pinned to the packed one, which the golden packed-K
example pins to the page: appending the same tokens through both layouts must
give byte buffers that are the same array seen through the two shapes (the
packed view un-interleaved with numpy's own transpose), identical V, and
identical attention outputs.  A wrong stride or a swapped token/channel index
in either layout's offset fails the first check.
"""
import numpy as np
import pytest

import gk_inputs as gi
import oracle


def _append(w, c, st, k_layout):
    sh = oracle.make_shape(**gi.shape_dict(w, c), k_layout=k_layout)
    n = c.num_blocks * w.num_kv_heads * w.block_size * w.head_dim
    kb = [np.zeros(n, np.uint8) for _ in range(w.num_layers // 2)]
    vb = [np.zeros(n, np.uint8) for _ in range(w.num_layers // 2)]
    assert oracle.kv_append(sh, gi.bf16_bits(st["k_new"]), gi.bf16_bits(st["v_new"]), c.cos,
                            c.sin, c.k_scale, c.v_scale, c.upd_full, c.upd_swa, c.active, kb,
                            vb) == 0
    return sh, kb, vb


def _unpack(kbuf, nb, Hkv, B, D):
    """Packed bytes [nb, Hkv, B/2, D, 2] -> the unpacked array [nb, Hkv, B, D]."""
    return kbuf.reshape(nb, Hkv, B // 2, D, 2).transpose(0, 1, 2, 4, 3).reshape(-1)


@pytest.mark.parametrize("name", ["tiny", "block16_small", "gk120b_rank_small"])
def test_append_unpacked_is_packed_uninterleaved(name):
    w = gi.get(name)
    c = gi.make_control(w)
    st = gi.make_step(w, "cpu")
    _, kp, vp = _append(w, c, st, 0)
    _, ku, vu = _append(w, c, st, 1)
    wrote = 0
    for j in range(w.num_layers // 2):
        assert np.array_equal(_unpack(kp[j], c.num_blocks, w.num_kv_heads, w.block_size,
                                      w.head_dim), ku[j]), j
        assert np.array_equal(vp[j], vu[j]), j
        wrote += int(np.count_nonzero(ku[j]))
    assert wrote > 0


def test_unpacked_offset_is_row_major_index():
    """Element (pb, h, t, e) of the unpacked K lands at numpy's row-major index
    of [nb, Hkv, B, D]: the appended row of one token sits in one D-byte run."""
    w = gi.get("tiny")
    c = gi.make_control(w)
    st = gi.make_step(w, "cpu")
    _, ku, _ = _append(w, c, st, 1)
    B, Hkv, D = w.block_size, w.num_kv_heads, w.head_dim
    b = int(np.nonzero(c.active)[0][0])
    slot = int(c.upd_full[b])                       # layer 1 (full) uses buffer 0
    pb, t = divmod(slot, B)
    for h in range(Hkv):
        lo = np.ravel_multi_index((pb, h, t, 0), (c.num_blocks, Hkv, B, D))
        row = ku[0][lo:lo + D]
        assert np.count_nonzero(row) > D // 2      # the token's codes, not padding


@pytest.mark.parametrize("name", ["tiny", "block16_small"])
def test_attention_same_in_both_layouts(name):
    w = gi.get(name)
    c = gi.make_control(w)
    st = gi.make_step(w, "cpu")
    cache = gi.make_cache(w, c, "cpu")
    kpk = [b[0].numpy().reshape(-1).copy() for b in cache]
    vpk = [b[1].numpy().reshape(-1).copy() for b in cache]
    kun = [_unpack(k, c.num_blocks, w.num_kv_heads, w.block_size, w.head_dim).copy() for k in kpk]
    q = gi.bf16_bits(st["q"])
    args = (c.k_scale, c.v_scale, c.cos, c.sin, c.bt_full, c.bt_swa, c.pos, c.pos_w, c.active)
    o0, s0 = oracle.decode_attn_stack(oracle.make_shape(**gi.shape_dict(w, c), k_layout=0), q,
                                      kpk, vpk, *args)
    o1, s1 = oracle.decode_attn_stack(oracle.make_shape(**gi.shape_dict(w, c), k_layout=1), q,
                                      kun, vpk, *args)
    assert s0 == 0 and s1 == 0
    assert np.array_equal(o0, o1)
    assert np.abs(o0).max() > 0
