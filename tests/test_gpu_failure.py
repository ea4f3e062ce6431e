"""Failure detection on the GPU without a fault: the bounded barrier wait that
every attention pipeline stage uses runs into its limit on a barrier phase
that nothing completes, reports GK_DEVERR_TIMEOUT through the error word, and
the context keeps working."""
import time

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


def test_bounded_wait_times_out_and_reports():
    t0 = time.perf_counter()
    bits = gk.gk_selftest_wait_timeout(20_000_000)      # 20 ms
    dt = time.perf_counter() - t0
    assert bits == gk.GK_DEVERR_TIMEOUT
    assert 0.015 < dt < 2.0
    assert gk.gk_read_device_error() == 0               # cleared


def test_context_usable_after_timeout():
    gk.gk_selftest_wait_timeout(1_000_000)
    w = gi.get("tiny")
    c = gi.make_control(w)
    st = gi.make_step(w, "cpu")
    cache = gi.make_cache(w, c, "cpu")
    ref, _, _ = tl.oracle_step(w, c, st, cache)
    g = tl.GpuStep(w, c, st, cache)
    g.append()
    g.attention()
    torch.cuda.synchronize()
    assert gk.gk_read_device_error() == 0
    tl.check_out(g.out.float().cpu().numpy().astype(np.float64),
                 g.out_f32.cpu().numpy().astype(np.float64), ref, "after timeout")
