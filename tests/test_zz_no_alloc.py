"""gk_decode_attn_stack_static: decode attention for callers that cannot
allocate device memory (a framework that budgets every device byte before the
first step, a plugin boundary without a device allocator, a step that must not
risk cudaMalloc's synchronisation or failure).  It runs on the library's own
fixed scratch array instead of a caller workspace.

Checked through the C ABI against the workspace entry point and against the
oracle on the same inputs, on two calls in a row (the second call reuses the
array the first one left behind), within the parity tests' tolerance; and once
at the 36-layer batch-64 size, where the fixed array holds fewer split-KV
records than the recommended workspace, against the oracle on every output
element.  Works alone in a fresh process and after the other tests.
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
    ora, _, _ = tl.oracle_step(w, c, st, cache)
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
        tl.check_out(_f64(out), _f64(out_f32), ref, f"{name} static call {call} vs workspace")
        tl.check_out(_f64(out), _f64(out_f32), ora, f"{name} static call {call} vs oracle")


def test_static_scratch_full_size_against_the_oracle():
    """36 layers, batch 64, contexts U{1024..8192}: the recommended workspace
    is larger than the fixed array, so the planner runs with fewer split-KV
    records than it would choose (longer chunks); every output element still
    meets the tolerance against the oracle."""
    w = gi.get("gptoss_b64")
    c = gi.make_control(w)
    st = gi.make_step(w, "cuda")
    cache = gi.make_cache(w, c, "cuda")
    pre = [b.clone() for b in cache]
    g = tl.GpuStep(w, c, st, cache)
    assert gk.gk_attn_workspace_bytes(g.shape) > (16 << 20) >= gk.gk_attn_workspace_min_bytes(g.shape)
    g.append()
    out = torch.full_like(g.out, float("nan"))
    out_f32 = torch.full_like(g.out_f32, float("nan"))
    gk.gk_decode_attn_stack_static(g.shape, g.q, g.kv, g.k_scale, g.v_scale, g.cos, g.sin,
                                   g.bt_full, g.bt_swa, g.pos, g.pos_w, g.active, out, out_f32)
    torch.cuda.synchronize()
    assert gk.gk_read_device_error() == 0
    o, of = _f64(out), _f64(out_f32)
    del g, cache, out, out_f32
    host = {k: gi.bf16_bits(v) for k, v in st.items()}
    ref = tl.oracle_full_output(w, c, host, pre)
    tl.check_out(o, of, ref, "gptoss_b64 static whole output")


def test_static_scratch_holds_every_accepted_shape():
    """The fixed array holds the minimum workspace of the largest shape the
    library accepts (128 layers, batch 8192, 64 kv heads, 1024-token blocks),
    so the no-allocation entry point refuses no valid shape for lack of room
    (a larger array only buys more split-KV records); a shape the library
    does not support is refused on the host before anything is launched."""
    sh = gk.Shape.make(num_layers=128, batch=8192, num_q_heads=512, num_kv_heads=64, head_dim=64,
                       block_size=1024, num_blocks=1 << 16, window=128, max_blocks_full=1024,
                       max_blocks_swa=2)
    need = gk.gk_attn_workspace_min_bytes(sh)
    assert 0 < need <= (16 << 20)
    bad = gk.Shape.make(num_layers=4, batch=2, num_q_heads=16, num_kv_heads=2, head_dim=128,
                        block_size=32, num_blocks=64, window=128, max_blocks_full=8,
                        max_blocks_swa=5)
    good = ctypes.c_void_p(0x10000)
    arr = (ctypes.c_void_p * 64)(*([0x10000] * 64))
    kvs = gk.KvCacheC(k_bufs=ctypes.cast(arr, ctypes.c_void_p),
                      v_bufs=ctypes.cast(arr, ctypes.c_void_p), k_layout=gk.GK_K_PACKED)
    st = gk.lib().gk_decode_attn_stack_static(ctypes.byref(bad), good, ctypes.byref(kvs),
                                              *([good] * 9), None, good, None, None)
    assert st == gk.GK_ERR_UNSUPPORTED
