"""The decode step captured once in a CUDA graph and replayed: the append,
planner and attention launches (chained by programmatic dependent launch)
replay with results bit-identical to direct calls.  Capturing the step
removes the per-step host launch cost for serving loops."""
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


@pytest.mark.parametrize("name,fused", [("gptoss_small", False), ("long_small", False),
                                        ("gptoss_small", True)])
def test_graph_replay_matches_direct_calls(name, fused):
    w = gi.get(name)
    c = gi.make_control(w)
    st = gi.make_step(w, "cpu")
    cache = gi.make_cache(w, c, "cpu")
    direct = tl.GpuStep(w, c, st, [b.clone() for b in cache])
    if fused:
        direct.step()
    else:
        direct.append()
        direct.attention()
    torch.cuda.synchronize()

    g = tl.GpuStep(w, c, st, [b.clone() for b in cache])
    g.attention()                      # first call on the device: setup outside the capture
    torch.cuda.synchronize()
    g.out.zero_()
    g.out_f32.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        if fused:
            g.step()
        else:
            g.append()
            g.attention()
    for _ in range(3):                 # replays re-append the same codes: idempotent
        graph.replay()
    torch.cuda.synchronize()
    assert gk.gk_read_device_error() == 0
    for a, b in zip(direct.cache, g.cache):
        assert torch.equal(a, b)
    assert torch.equal(direct.out, g.out) and torch.equal(direct.out_f32, g.out_f32)
    ref, _, _ = tl.oracle_step(w, c, st, cache)
    tl.check_out(g.out.float().cpu().numpy().astype(np.float64),
                 g.out_f32.cpu().numpy().astype(np.float64), ref, f"{name} graph")
