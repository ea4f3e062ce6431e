"""gk_decode_attn_stack_static: decode attention for callers that cannot
allocate device memory (a framework that budgets every device byte before the
first step, a plugin boundary without a device allocator, a step that must not
risk cudaMalloc's synchronisation or failure).  It runs on the library's own
fixed scratch array instead of a caller workspace.

Checked through the C ABI against the workspace entry point on the same
inputs, on two calls in a row (the second call reuses the array the first one
left behind), within the parity tests' tolerance.  Works alone in a fresh
process and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import gk_inputs as gi
import gk_testlib as tl
import paged_fp8_kv_gk_gb300 as gk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    gk.lib()
    gk.gk_read_device_error(clear=True)


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("name", ["gptoss_small", "long_small", "ragged_small"])
def test_static_scratch_matches_workspace_entry_point(name):
    w = gi.get(name)
    c = gi.make_control(w)
    st = gi.make_step(w, "cpu")
    cache = gi.make_cache(w, c, "cpu")
    g = tl.GpuStep(w, c, st, cache)
    g.append()
    g.attention()                       # existing entry point, caller workspace
    torch.cuda.synchronize()
    ref = _f64(g.out_f32)
    for call in range(2):
        out = torch.full_like(g.out, float("nan"))
        out_f32 = torch.full_like(g.out_f32, float("nan"))
        gk.gk_decode_attn_stack_static(g.shape, g.q, g.kv, g.k_scale, g.v_scale, g.cos,
                                       g.sin, g.bt_full, g.bt_swa, g.pos, g.pos_w, g.active, out,
                                       out_f32)
        torch.cuda.synchronize()
        assert gk.gk_read_device_error() == 0
        tl.check_out(_f64(out), _f64(out_f32), ref, f"{name} static call {call}")


def test_static_scratch_rejects_shapes_beyond_its_size():
    """A shape whose minimum workspace exceeds the fixed array is refused on
    the host with GK_ERR_WORKSPACE; nothing is launched."""
    sh = gk.Shape.make(num_layers=128, batch=8192, num_q_heads=512, num_kv_heads=64, head_dim=64,
                       block_size=32, num_blocks=1 << 16, window=128, max_blocks_full=64,
                       max_blocks_swa=5)
    assert gk.gk_attn_workspace_min_bytes(sh) > (16 << 20)
    good = ctypes.c_void_p(0x10000)
    arr = (ctypes.c_void_p * 64)(*([0x10000] * 64))
    kvs = gk.KvCacheC(k_bufs=ctypes.cast(arr, ctypes.c_void_p),
                      v_bufs=ctypes.cast(arr, ctypes.c_void_p), k_layout=gk.GK_K_PACKED)
    st = gk.lib().gk_decode_attn_stack_static(ctypes.byref(sh), good, ctypes.byref(kvs),
                                              *([good] * 9), None, good, None, None)
    assert st == gk.GK_ERR_WORKSPACE
