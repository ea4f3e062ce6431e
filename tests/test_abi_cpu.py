"""The C-ABI library builds, loads and exports every symbol include/gk.h
declares; host-side argument validation returns the documented status before
anything reaches the device.  No compute call is made (CPU only)."""
import ctypes

import pytest

import gk_inputs as gi
import paged_fp8_kv_gk_gb300 as gk

EXPECTED = {"gk_kv_append", "gk_attn_workspace_bytes", "gk_attn_workspace_min_bytes",
            "gk_decode_attn_stack", "gk_e4m3_quantize", "gk_read_device_error",
            "gk_status_str", "gk_abi_version", "gk_decode_attn_stack_static", "gk_kv_budget",
            "gk_decode_step"}


def test_header_declares_the_boundary():
    assert set(gk.declared_functions()) == EXPECTED


def test_library_exports_every_declared_symbol():
    L = gk.lib()
    for name in gk.declared_functions():
        assert hasattr(L, name), name
        assert callable(getattr(gk, name)), name


def test_version_and_status_strings():
    assert gk.gk_abi_version() == 1
    names = [gk.gk_status_str(i) for i in range(7)]
    assert names == ["GK_OK", "GK_ERR_INVALID_ARG", "GK_ERR_UNSUPPORTED", "GK_ERR_WORKSPACE",
                     "GK_ERR_CUDA", "GK_ERR_DEVICE_BOUNDS", "GK_ERR_BUDGET"]
    assert gk.gk_status_str(99) == "GK_ERR_UNKNOWN"


def _shape(name="gptoss_b64", **over):
    w = gi.get(name)
    c = gi.make_control(w)       # host control tensors only; cheap at full size
    d = gi.shape_dict(w, c)
    d.update(over)
    return gk.Shape.make(**d)


@pytest.mark.parametrize("name", ["tiny", "gptoss_b64", "long_ctx", "ragged_b256", "swa_b512"])
def test_workspace_sizes(name):
    sh = _shape(name)
    mn, rec = gk.gk_attn_workspace_min_bytes(sh), gk.gk_attn_workspace_bytes(sh)
    assert 0 < mn <= rec
    assert mn % 256 == 0 and rec % 256 == 0
    if name == "swa_b512":     # contexts <= 512 never split: no partial capacity
        assert rec == mn


@pytest.mark.parametrize("over,status", [
    (dict(num_layers=3), gk.GK_ERR_INVALID_ARG),
    (dict(num_layers=0), gk.GK_ERR_INVALID_ARG),
    (dict(batch=0), gk.GK_ERR_INVALID_ARG),
    (dict(num_q_heads=60), gk.GK_ERR_INVALID_ARG),
    (dict(block_size=31), gk.GK_ERR_INVALID_ARG),
    (dict(max_blocks_swa=4), gk.GK_ERR_INVALID_ARG),
    (dict(head_dim=128), gk.GK_ERR_UNSUPPORTED),
    (dict(num_q_heads=32), gk.GK_ERR_UNSUPPORTED),
    (dict(block_size=48), gk.GK_ERR_UNSUPPORTED),
    (dict(num_layers=130), gk.GK_ERR_UNSUPPORTED),
    (dict(batch=9000), gk.GK_ERR_UNSUPPORTED),
])
def test_shape_validation(over, status):
    sh = _shape("gptoss_b64", **over)
    L = gk.lib()
    assert L.gk_attn_workspace_bytes(ctypes.byref(sh), None) == 0
    fake = ctypes.c_void_p(0x10000)
    ptrs = (ctypes.c_void_p * 64)(*([0x10000] * 64))
    args = [fake] * 9 + [ctypes.cast(ptrs, ctypes.c_void_p)] * 2 + [None]
    assert L.gk_kv_append(ctypes.byref(sh), *args) == status


def test_null_and_alignment_checks_before_launch():
    sh = _shape("gptoss_b64")
    L = gk.lib()
    good = ctypes.c_void_p(0x10000)
    ptrs = ctypes.cast((ctypes.c_void_p * 64)(*([0x10000] * 64)), ctypes.c_void_p)
    # append: one null tensor pointer
    args = [good] * 9 + [ptrs, ptrs, None]
    for i in range(9):
        a = list(args)
        a[i] = None
        assert L.gk_kv_append(ctypes.byref(sh), *a) == gk.GK_ERR_INVALID_ARG
    # append: misaligned k_new
    a = list(args)
    a[0] = ctypes.c_void_p(0x10002)
    assert L.gk_kv_append(ctypes.byref(sh), *a) == gk.GK_ERR_INVALID_ARG
    # append: a null group buffer pointer
    bad = (ctypes.c_void_p * 64)(*([0x10000] * 64))
    bad[5] = None
    a = list(args)
    a[9] = ctypes.cast(bad, ctypes.c_void_p)
    assert L.gk_kv_append(ctypes.byref(sh), *a) == gk.GK_ERR_INVALID_ARG

    # attention: nulls, then workspace checks (all before any launch)
    att = [good, ptrs, ptrs] + [good] * 10 + [None, good]   # q..out, out_f32, workspace
    ws_min = L.gk_attn_workspace_min_bytes(ctypes.byref(sh))

    def call(a, nbytes):
        return L.gk_decode_attn_stack(ctypes.byref(sh), *a, nbytes, None)

    for i in range(13):
        a = list(att)
        a[i] = None
        assert call(a, ws_min) == gk.GK_ERR_INVALID_ARG, i
    a = list(att)
    a[14] = None
    assert call(a, ws_min) == gk.GK_ERR_WORKSPACE
    a = list(att)
    a[14] = ctypes.c_void_p(0x10080)          # not 256-byte aligned
    assert call(a, ws_min) == gk.GK_ERR_WORKSPACE
    assert call(att, ws_min - 256) == gk.GK_ERR_WORKSPACE
    a = list(att)
    a[13] = ctypes.c_void_p(0x10004)          # misaligned out_f32
    assert call(a, ws_min) == gk.GK_ERR_INVALID_ARG
    assert L.gk_e4m3_quantize(None, ctypes.c_float(1.0), None, -1, None) == gk.GK_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors():
    import torch
    sh = _shape("tiny")
    t = torch.zeros(16, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        gk.gk_kv_append(sh, t, t, t, t, t, t, t, t, t, [t], [t], stream=0)


def test_testing_header_symbol_exported_and_validates():
    L = gk.lib()
    assert hasattr(L, "gk_selftest_wait_timeout")
    b = ctypes.c_uint32()
    assert L.gk_selftest_wait_timeout(10, None, ctypes.byref(b)) == gk.GK_ERR_INVALID_ARG
    assert L.gk_selftest_wait_timeout(10 ** 10, None, ctypes.byref(b)) == gk.GK_ERR_INVALID_ARG
    assert L.gk_selftest_wait_timeout(10 ** 6, None, None) == gk.GK_ERR_INVALID_ARG
