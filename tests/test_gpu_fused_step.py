"""GPU parity of the fused decode step (gk_decode_step): the same KV bytes as
the separate append and the same outputs as the separate attention, checked
against the oracle exactly as the two-call path is."""
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


@pytest.mark.parametrize("name", ["tiny", "gptoss_small", "long_small", "ragged_small",
                                  "swa_small_sat", "block16_small"])
def test_fused_step_parity(name):
    w = gi.get(name)
    c = gi.make_control(w)
    st = gi.make_step(w, "cpu")
    cache = gi.make_cache(w, c, "cpu")
    ref, kb_ref, vb_ref = tl.oracle_step(w, c, st, cache)
    g = tl.GpuStep(w, c, st, cache)
    g.step()
    torch.cuda.synchronize()
    assert gk.gk_read_device_error() == 0
    for j in range(len(g.cache)):
        assert np.array_equal(g.cache[j][0].cpu().numpy().reshape(-1), kb_ref[j]), ("K", j)
        assert np.array_equal(g.cache[j][1].cpu().numpy().reshape(-1), vb_ref[j]), ("V", j)
    out, of = _f64(g.out), _f64(g.out_f32)
    tl.check_out(out, of, ref, name + "/fused")
    assert (out[:, c.active == 0] == 0).all()


def test_fused_equals_two_calls_bitwise():
    w = gi.get("long_small")
    c = gi.make_control(w)
    st = gi.make_step(w, "cpu")
    cache = gi.make_cache(w, c, "cpu")
    a = tl.GpuStep(w, c, st, [b.clone() for b in cache])
    a.append()
    a.attention()
    b = tl.GpuStep(w, c, st, [x.clone() for x in cache])
    b.step()
    torch.cuda.synchronize()
    for x, y in zip(a.cache, b.cache):
        assert torch.equal(x, y)
    assert torch.equal(a.out, b.out) and torch.equal(a.out_f32, b.out_f32)


@pytest.mark.parametrize("name", ["gptoss_b64", "swa_b512", "long_ctx"])
def test_fused_step_full_size(name):
    """gk_decode_step at full size: every appended KV byte bit-exact and every
    output element against the oracle."""
    w = gi.get(name)
    c = gi.make_control(w)
    st = gi.make_step(w, "cuda")
    cache = gi.make_cache(w, c, "cuda")
    pre = [x.clone() for x in cache]
    g = tl.GpuStep(w, c, st, cache)
    g.step()
    torch.cuda.synchronize()
    assert gk.gk_read_device_error() == 0
    kc_d, vc_d = tl.device_appended_codes(g)
    kc_o, vc_o = tl.oracle_appended_codes(w, c, st)
    act = c.active == 1
    assert np.array_equal(kc_d[:, act], kc_o[:, act]) and np.array_equal(vc_d[:, act], vc_o[:, act])
    out, of = _f64(g.out), _f64(g.out_f32)
    del g, cache
    host = {k: gi.bf16_bits(v) for k, v in st.items()}
    ref = tl.oracle_full_output(w, c, host, pre)
    tl.check_out(out, of, ref, f"{name} gk_decode_step whole output")
