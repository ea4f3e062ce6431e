"""Split-KV (flash-decoding) combine at fixed chunk counts: the test hook
gk_selftest_decode_attn_split (include/gk_testing.h) fixes the chunk length,
so rows of 300, 1000, 3500, 32768 and 32257 keys take 1, 2, 7, 64 and 64
chunks at 512 tokens (64 is the cap per (layer, row, kv head); the last row's
final chunk holds a single key), fewer at longer chunks.  Every output element
is compared with the oracle, with and without attention sinks."""
import numpy as np
import pytest
import torch

import gk_inputs as gi
import gk_testlib as tl
import paged_fp8_kv_gk_gb300 as gk

pytestmark = pytest.mark.gpu

_ORACLE = {}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    gk.lib()
    gk.gk_read_device_error(clear=True)


def _inputs(with_sinks):
    w = gi.get("split_counts_small")
    c = gi.make_control(w)
    st = gi.make_step(w, "cpu")
    cache = gi.make_cache(w, c, "cpu")
    sinks = gi.make_sinks(w) if with_sinks else None
    if with_sinks not in _ORACLE:
        _ORACLE[with_sinks] = tl.oracle_step(w, c, st, cache, sinks=sinks)[0]
    return w, c, st, cache, sinks, _ORACLE[with_sinks]


@pytest.mark.parametrize("with_sinks", [False, True])
@pytest.mark.parametrize("split", [512, 1024, 4096, 65536])
def test_forced_split_counts(split, with_sinks):
    w, c, st, cache, sinks, ref = _inputs(with_sinks)
    counts = [-(-int(L) // split) for L in c.lengths]
    if split == 512:
        assert counts == [1, 2, 7, 64, 64]
    g = tl.GpuStep(w, c, st, cache, sinks=sinks)
    g.append()
    g.out.fill_(float("nan"))
    gk.gk_selftest_decode_attn_split(g.shape, g.q, g.kv, g.k_scale, g.v_scale, g.cos, g.sin,
                                     g.bt_full, g.bt_swa, g.pos, g.pos_w, g.active, g.out,
                                     g.out_f32, g.workspace, split, sinks=g.sinks)
    torch.cuda.synchronize()
    assert gk.gk_read_device_error() == 0
    hdr = g.workspace[:256].view(torch.int32).cpu().numpy()
    assert hdr[4] == split and hdr[7] == 0, hdr[:8]
    assert hdr[6] == sum(n for n in counts if n > 1), (hdr[6], counts)
    out = g.out.float().cpu().numpy().astype(np.float64)
    of = g.out_f32.cpu().numpy().astype(np.float64)
    tl.check_out(out, of, ref, f"split {split} sinks {with_sinks}")


def test_split_length_raised_past_the_chunk_cap():
    """A row of 40000 keys would need 79 chunks of 512: the length is raised
    to 1024 (40 chunks), and the output still meets the tolerance."""
    w = gi.get("split_counts_small").replace(name="split_cap_small", batch=2,
                                             lengths="fixed:40000,700", seed=34)
    c = gi.make_control(w)
    st = gi.make_step(w, "cpu")
    cache = gi.make_cache(w, c, "cpu")
    ref, _, _ = tl.oracle_step(w, c, st, cache)
    g = tl.GpuStep(w, c, st, cache)
    g.append()
    gk.gk_selftest_decode_attn_split(g.shape, g.q, g.kv, g.k_scale, g.v_scale, g.cos, g.sin,
                                     g.bt_full, g.bt_swa, g.pos, g.pos_w, g.active, g.out,
                                     g.out_f32, g.workspace, 512)
    torch.cuda.synchronize()
    assert gk.gk_read_device_error() == 0
    hdr = g.workspace[:256].view(torch.int32).cpu().numpy()
    assert hdr[4] == 1024 and hdr[6] == 40, hdr[:8]
    tl.check_out(g.out.float().cpu().numpy().astype(np.float64),
                 g.out_f32.cpu().numpy().astype(np.float64), ref, "raised split")
