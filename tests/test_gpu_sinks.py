"""GPU parity of the optional attention sinks (GPT-OSS per-head sink logits;
not on the pages): out = sum_t e^(s_t) v_t / (sum_t e^(s_t) + e^(sink)).

Sinks are N(0, 2) with some heads at +12 (the sink dominates: the overflow-safe
branch of the normalisation) and some at -30 (it vanishes).  Checked on small
workloads element by element (unsplit and split-KV rows), on the fused step
(bit-identical to append + attention), and on sampled rows at full size.
"""
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


@pytest.mark.parametrize("name", ["tiny", "gptoss_small", "long_small", "swa_small_peaky",
                                  "block16_small", "gk120b_rank_small"])
def test_sinks_parity(name):
    w = gi.get(name)
    c = gi.make_control(w)
    st = gi.make_step(w, "cpu")
    cache = gi.make_cache(w, c, "cpu")
    sinks = gi.make_sinks(w)
    ref, _, _ = tl.oracle_step(w, c, st, cache, sinks=sinks)
    g = tl.GpuStep(w, c, st, cache, sinks=sinks)
    g.append()
    g.attention()
    torch.cuda.synchronize()
    assert gk.gk_read_device_error() == 0
    tl.check_out(_f64(g.out), _f64(g.out_f32), ref, f"{name} sinks")
    # the sink-free output differs wherever a sink is not negligible
    plain, _, _ = tl.oracle_step(w, c, st, cache)
    act = c.active == 1
    assert np.abs(plain[:, act] - ref[:, act]).max() > 1e-2


def test_sinks_split_and_unsplit_agree():
    w = gi.get("long_small")
    c = gi.make_control(w)
    st = gi.make_step(w, "cpu")
    cache = gi.make_cache(w, c, "cpu")
    sinks = gi.make_sinks(w, seed=1)
    g = tl.GpuStep(w, c, st, cache, sinks=sinks)
    g.append()
    g.attention()
    split = g.out_f32.clone()
    ws_min = torch.empty(gk.gk_attn_workspace_min_bytes(g.shape), dtype=torch.uint8,
                         device="cuda")
    g.attention(workspace=ws_min)
    torch.cuda.synchronize()
    assert gk.gk_read_device_error() == 0
    d = (split - g.out_f32).abs().max().item()
    assert d <= 1e-4, d


def test_fused_step_with_sinks_equals_two_calls():
    w = gi.get("gptoss_small")
    c = gi.make_control(w)
    st = gi.make_step(w, "cpu")
    cache = gi.make_cache(w, c, "cpu")
    sinks = gi.make_sinks(w)
    a = tl.GpuStep(w, c, st, [x.clone() for x in cache], sinks=sinks)
    a.append()
    a.attention()
    b = tl.GpuStep(w, c, st, [x.clone() for x in cache], sinks=sinks)
    b.step()
    torch.cuda.synchronize()
    for x, y in zip(a.cache, b.cache):
        assert torch.equal(x, y)
    assert torch.equal(a.out, b.out) and torch.equal(a.out_f32, b.out_f32)


def test_full_size_sinks_whole_output():
    """Attention sinks on the 36-layer batch-64 workload: every output element
    against the oracle."""
    w = gi.get("gptoss_b64")
    c = gi.make_control(w)
    st = gi.make_step(w, "cuda")
    cache = gi.make_cache(w, c, "cuda")
    pre = [x.clone() for x in cache]
    sinks = gi.make_sinks(w)
    g = tl.GpuStep(w, c, st, cache, sinks=sinks)
    g.append()
    g.attention()
    torch.cuda.synchronize()
    assert gk.gk_read_device_error() == 0
    out, of = _f64(g.out), _f64(g.out_f32)
    del g, cache
    host = {k: gi.bf16_bits(v) for k, v in st.items()}
    ref = tl.oracle_full_output(w, c, host, pre, sinks=sinks)
    tl.check_out(out, of, ref, "sinks whole output")
