"""The C-ABI library builds, loads and exports every symbol include/gk.h
declares; host-side argument validation returns the documented status before
anything reaches the device.  No compute call is made (CPU only).

The validation tests hand the library fake device addresses together with one
invalid argument; they run only where no CUDA device is visible, so that a
validation bug can never turn one of them into a launch on real memory."""
import ctypes

import pytest
import torch

import gk_inputs as gi
import paged_fp8_kv_gk_gb300 as gk

EXPECTED = {"gk_kv_append", "gk_attn_workspace_bytes", "gk_attn_workspace_min_bytes",
            "gk_decode_attn_stack", "gk_e4m3_quantize", "gk_read_device_error",
            "gk_status_str", "gk_abi_version", "gk_decode_attn_stack_static", "gk_kv_budget",
            "gk_decode_step", "gk_kv_regions", "gk_kv_ingest", "gk_di_blocks"}


def test_header_declares_the_boundary():
    assert set(gk.declared_functions()) == EXPECTED


def test_library_exports_every_declared_symbol():
    L = gk.lib()
    for name in gk.declared_functions():
        assert hasattr(L, name), name
        assert callable(getattr(gk, name)), name


no_device = pytest.mark.skipif(torch.cuda.is_available(),
                               reason="fake device addresses: run only without a GPU")

FAKE = 0x10000


def _kv_struct(form="per_group", k_layout=gk.GK_K_PACKED, n=64, bad_index=None, k_addr=FAKE,
               v_addr=FAKE):
    """A gk_kv_cache over fake addresses (kept alive by the returned tuple)."""
    c = gk.KvCacheC(k_layout=k_layout)
    arrs = ()
    if form in ("per_group", "both"):
        ka = (ctypes.c_void_p * n)(*([FAKE] * n))
        va = (ctypes.c_void_p * n)(*([FAKE] * n))
        if bad_index is not None:
            ka[bad_index] = None
        c.k_bufs = ctypes.cast(ka, ctypes.c_void_p)
        c.v_bufs = ctypes.cast(va, ctypes.c_void_p)
        arrs = (ka, va)
    if form in ("stacked", "both"):
        c.k_cache = k_addr
        c.v_cache = v_addr
    return c, arrs


def test_version_and_status_strings():
    assert gk.gk_abi_version() == 3
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


@no_device
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
    fake = ctypes.c_void_p(FAKE)
    kvs, keep = _kv_struct()
    args = [fake] * 9 + [ctypes.byref(kvs), None]
    assert L.gk_kv_append(ctypes.byref(sh), *args) == status


@no_device
def test_null_and_alignment_checks_before_launch():
    sh = _shape("gptoss_b64")
    L = gk.lib()
    good = ctypes.c_void_p(FAKE)
    kvs, keep = _kv_struct()
    kv = ctypes.byref(kvs)
    # append: one null tensor pointer
    args = [good] * 9 + [kv, None]
    for i in range(9):
        a = list(args)
        a[i] = None
        assert L.gk_kv_append(ctypes.byref(sh), *a) == gk.GK_ERR_INVALID_ARG
    # append: misaligned k_new
    a = list(args)
    a[0] = ctypes.c_void_p(0x10002)
    assert L.gk_kv_append(ctypes.byref(sh), *a) == gk.GK_ERR_INVALID_ARG
    # append: a null group buffer pointer
    badkv, keep2 = _kv_struct(bad_index=5)
    a = list(args)
    a[9] = ctypes.byref(badkv)
    assert L.gk_kv_append(ctypes.byref(sh), *a) == gk.GK_ERR_INVALID_ARG

    # attention: nulls, then workspace checks (all before any launch)
    # q, kv, k_scale..active, sinks (optional), out, out_f32 (optional), workspace
    att = [good, kv] + [good] * 9 + [None, good, None, good]
    ws_min = L.gk_attn_workspace_min_bytes(ctypes.byref(sh))

    def call(a, nbytes):
        return L.gk_decode_attn_stack(ctypes.byref(sh), *a, nbytes, None)

    for i in list(range(11)) + [12]:
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
    a = list(att)
    a[11] = ctypes.c_void_p(0x10002)          # misaligned sinks
    assert call(a, ws_min) == gk.GK_ERR_INVALID_ARG
    assert L.gk_e4m3_quantize(None, ctypes.c_float(1.0), None, -1, None) == gk.GK_ERR_INVALID_ARG


@no_device
@pytest.mark.parametrize("case", ["both", "neither", "stacked_k_only", "layout_2",
                                  "stacked_misaligned", "per_group_null"])
def test_kv_form_exactly_one(case):
    """The cache descriptor must hold exactly one form ("Kernel contract": the
    kernel asserts that exactly one of per-group / stacked is present), with a
    known K layout; everything else is refused on the host."""
    sh = _shape("gptoss_b64")
    L = gk.lib()
    good = ctypes.c_void_p(FAKE)
    if case == "both":
        kvs, keep = _kv_struct("both")
    elif case == "neither":
        kvs, keep = _kv_struct("none")
    elif case == "stacked_k_only":
        kvs, keep = _kv_struct("stacked", v_addr=None)
    elif case == "layout_2":
        kvs, keep = _kv_struct("stacked", k_layout=2)
    elif case == "stacked_misaligned":
        kvs, keep = _kv_struct("stacked", k_addr=FAKE + 8)
    else:
        kvs, keep = _kv_struct("per_group", bad_index=17)
    assert L.gk_kv_append(ctypes.byref(sh), *([good] * 9), ctypes.byref(kvs), None) == \
        gk.GK_ERR_INVALID_ARG
    ws_min = L.gk_attn_workspace_min_bytes(ctypes.byref(sh))
    assert L.gk_decode_attn_stack(ctypes.byref(sh), good, ctypes.byref(kvs), *([good] * 9), None,
                                  good, None, good, ws_min, None) == gk.GK_ERR_INVALID_ARG


def test_binding_kv_forms_and_rank_inference():
    """KvCache: exactly one form; packed-ness from the ranks as the page's bind
    step infers it (k.dim() == v.dim() + 1); CPU tensors are refused."""
    v = torch.zeros(4, 1, 16, 64, dtype=torch.uint8)
    k_packed = torch.zeros(4, 1, 8, 64, 2, dtype=torch.uint8)
    assert gk.infer_k_layout(k_packed, v) == gk.GK_K_PACKED
    assert gk.infer_k_layout(v.clone(), v) == gk.GK_K_PLAIN
    with pytest.raises(ValueError):
        gk.infer_k_layout(torch.zeros(4, 1, 16, 64, 1, 1, dtype=torch.uint8), v)
    with pytest.raises(ValueError, match="exactly one"):
        gk.KvCache(k_bufs=[k_packed], v_bufs=[v], k_cache=k_packed, v_cache=v)
    with pytest.raises(ValueError, match="exactly one"):
        gk.KvCache()
    with pytest.raises(ValueError, match="rank"):
        gk.KvCache(k_bufs=[k_packed], v_bufs=[v], k_layout=gk.GK_K_PLAIN)
    with pytest.raises(ValueError, match="one K layout"):
        gk.KvCache(k_bufs=[k_packed, v.clone()], v_bufs=[v, v])
    with pytest.raises(ValueError, match="CUDA"):
        gk.KvCache(k_bufs=[k_packed], v_bufs=[v])


@no_device
def test_binding_refuses_cpu_tensors():
    sh = _shape("tiny")
    t = torch.zeros(16, dtype=torch.bfloat16)
    kv = gk.KvCache(k_bufs=[FAKE], v_bufs=[FAKE], k_layout=gk.GK_K_PACKED)
    with pytest.raises(ValueError, match="CUDA"):
        gk.gk_kv_append(sh, t, t, t, t, t, t, t, t, t, kv, stream=0)


def test_testing_header_symbol_exported_and_validates():
    L = gk.lib()
    assert hasattr(L, "gk_selftest_wait_timeout")
    b = ctypes.c_uint32()
    assert L.gk_selftest_wait_timeout(10, None, ctypes.byref(b)) == gk.GK_ERR_INVALID_ARG
    assert L.gk_selftest_wait_timeout(10 ** 10, None, ctypes.byref(b)) == gk.GK_ERR_INVALID_ARG
    assert L.gk_selftest_wait_timeout(10 ** 6, None, None) == gk.GK_ERR_INVALID_ARG


@no_device
def test_split_hook_exported_and_validates_the_length():
    """gk_selftest_decode_attn_split (include/gk_testing.h) refuses a split
    length that is not a power of two from 512 to 512 << 21 before anything
    else is looked at."""
    L = gk.lib()
    sh = gk.Shape.make(num_layers=4, batch=5, num_q_heads=64, num_kv_heads=8, head_dim=64,
                       block_size=32, num_blocks=4096, window=128, max_blocks_full=1024,
                       max_blocks_swa=5)
    kvs, arrs = _kv_struct()
    for bad in (0, -512, 256, 513, 1000, 3 << 9, 512 << 22):
        st = L.gk_selftest_decode_attn_split(ctypes.byref(sh), FAKE, ctypes.byref(kvs),
                                             *([FAKE] * 9), None, FAKE, None, FAKE, 1 << 30, bad,
                                             None)
        assert st == gk.GK_ERR_INVALID_ARG, bad
