"""GPU parity of the two KV forms and the two K layouts ("GPT-OSS-120B
giga-kernel decode", section "Kernel contract": per-group buffers or stacked
K_cache / V_cache, exactly one present, packed-ness read from the K rank;
section "KV-cache layout": packed K view or unpacked K).

  * unpacked K: append bytes bit-exact and outputs within the parity tolerance
    against the oracle run on the unpacked layout, on small workloads of every
    block size, and on sampled rows of the full-size 36-layer batch-64 workload;
  * stacked form: bit-identical KV and outputs to the per-group form (the
    same kernels reading the same bytes at other addresses), both K layouts;
  * the fused step on unpacked K: bit-identical to append + attention.
"""
import numpy as np
import pytest
import torch

import gk_inputs as gi
import gk_testlib as tl
import paged_fp8_kv_gk_gb300 as gk

pytestmark = pytest.mark.gpu

PLAIN = gk.GK_K_PLAIN
PACKED = gk.GK_K_PACKED


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    gk.lib()
    gk.gk_read_device_error(clear=True)
    yield
    torch.cuda.synchronize()


def _make_cpu(name):
    w = gi.get(name)
    c = gi.make_control(w)
    return w, c, gi.make_step(w, "cpu"), gi.make_cache(w, c, "cpu")


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("name", ["tiny", "gptoss_small", "long_small", "ragged_small",
                                  "swa_small", "swa_small_peaky", "block16_small",
                                  "block64_small", "gk120b_rank_small"])
def test_unpacked_k_parity(name):
    w, c, st, cache = _make_cpu(name)
    ref, kb_ref, vb_ref = tl.oracle_step(w, c, st, cache, k_layout=1)
    g = tl.GpuStep(w, c, st, cache, k_layout=PLAIN)
    g.append()
    g.attention()
    torch.cuda.synchronize()
    assert gk.gk_read_device_error() == 0
    for j in range(len(g.cache)):
        assert np.array_equal(g.cache[j][0].cpu().numpy().reshape(-1), kb_ref[j]), ("K", j)
        assert np.array_equal(g.cache[j][1].cpu().numpy().reshape(-1), vb_ref[j]), ("V", j)
    tl.check_out(_f64(g.out), _f64(g.out_f32), ref, f"{name} unpacked K")


@pytest.mark.parametrize("k_layout", [PACKED, PLAIN])
@pytest.mark.parametrize("name", ["gptoss_small", "block16_small", "long_small"])
def test_stacked_equals_per_group(name, k_layout):
    w, c, st, cache = _make_cpu(name)
    a = tl.GpuStep(w, c, st, cache, k_layout=k_layout, form="per_group")
    b = tl.GpuStep(w, c, st, cache, k_layout=k_layout, form="stacked")
    for g in (a, b):
        g.append()
        g.attention()
    torch.cuda.synchronize()
    assert gk.gk_read_device_error() == 0
    for j in range(len(a.cache)):
        assert torch.equal(a.cache[j], b.cache[j]), j
    assert torch.equal(a.out, b.out) and torch.equal(a.out_f32, b.out_f32)


def test_fused_step_unpacked_equals_two_calls():
    w, c, st, cache = _make_cpu("long_small")
    a = tl.GpuStep(w, c, st, [x.clone() for x in cache], k_layout=PLAIN)
    a.append()
    a.attention()
    b = tl.GpuStep(w, c, st, [x.clone() for x in cache], k_layout=PLAIN)
    b.step()
    torch.cuda.synchronize()
    assert gk.gk_read_device_error() == 0
    for x, y in zip(a.cache, b.cache):
        assert torch.equal(x, y)
    assert torch.equal(a.out, b.out) and torch.equal(a.out_f32, b.out_f32)


def test_full_size_unpacked_k_whole_output():
    """Unpacked K in the stacked form on the 36-layer batch-64 workload: every
    appended byte bit-exact and every output element against the oracle."""
    name = "gptoss_b64"
    w = gi.get(name)
    c = gi.make_control(w)
    st = gi.make_step(w, "cuda")
    cache = gi.make_cache(w, c, "cuda")
    pre = [x.clone() for x in cache]
    g = tl.GpuStep(w, c, st, cache, k_layout=PLAIN, form="stacked")
    del cache
    g.append()
    g.attention()
    torch.cuda.synchronize()
    assert gk.gk_read_device_error() == 0
    kc_d, vc_d = tl.device_appended_codes(g)
    kc_o, vc_o = tl.oracle_appended_codes(w, c, st, k_layout=1)
    act = c.active == 1
    assert np.array_equal(kc_d[:, act], kc_o[:, act])
    assert np.array_equal(vc_d[:, act], vc_o[:, act])
    out, of = _f64(g.out), _f64(g.out_f32)
    del g
    host = {k: gi.bf16_bits(v) for k, v in st.items()}
    ref = tl.oracle_full_output(w, c, host, pre, k_layout=1)
    tl.check_out(out, of, ref, f"{name} unpacked K whole output")
