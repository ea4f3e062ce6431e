"""Back-to-back calls on one stream, nothing launched between them: each
call's outputs are exactly those of the same call run on its own.

The planner, the attention grid and the split-KV combine are chained by
programmatic dependent launches; a later call's planner rewrites the work
queue in the shared workspace, so it must not start while an earlier call's
attention grid still takes units from it.  Two alternating inputs (different
q, and for gk_decode_step different new tokens appended at the same
slots) make any unit done with the other call's arguments, or skipped, show
up as a mismatch or a NaN left in a NaN-filled output.  Run with and without
partial records (a workload whose rows can split, and one whose rows cannot),
with gk_decode_attn_stack and with gk_decode_step."""
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


def _steps(w):
    """Two input sets of one workload (the second: other q, k and v)."""
    a = gi.make_step(w, "cuda")
    b = gi.make_step(w.replace(seed=w.seed + 1000), "cuda")
    return a, b


@pytest.mark.parametrize("name,ws", [("swa_b128", "recommended"), ("gptoss_b16", "recommended"),
                                     ("gptoss_b8_8k", "minimum")])
@pytest.mark.parametrize("fused", [False, True])
def test_back_to_back_calls_match_single_calls(name, ws, fused):
    """The minimum workspace has no room for partial records: every row is
    one unit of 8192 keys, so warps are still deep in their units when the
    next call's planner could start (the case that would expose it)."""
    w = gi.get(name)
    c = gi.make_control(w)
    sa, sb = _steps(w)
    cache = gi.make_cache(w, c, "cuda")
    g = tl.GpuStep(w, c, sa, cache)
    if ws == "minimum":
        g.workspace = torch.empty(gk.gk_attn_workspace_min_bytes(g.shape), dtype=torch.uint8,
                                  device="cuda")
    reps = 6

    def call(st, out):
        if fused:
            gk.gk_decode_step(g.shape, st["q"], st["k_new"], st["v_new"], g.cos, g.sin, g.k_scale,
                              g.v_scale, g.upd_full, g.upd_swa, g.bt_full, g.bt_swa, g.pos,
                              g.pos_w, g.active, g.kv, out, None, g.workspace)
        else:
            gk.gk_decode_attn_stack(g.shape, st["q"], g.kv, g.k_scale, g.v_scale, g.cos, g.sin,
                                    g.bt_full, g.bt_swa, g.pos, g.pos_w, g.active, out, None,
                                    g.workspace)

    # references: each call alone.  gk_decode_step appends its own set's new
    # token before attending; the attention-only calls read the cache as the
    # append of set a left it.
    if not fused:
        gk.gk_kv_append(g.shape, sa["k_new"], sa["v_new"], g.cos, g.sin, g.k_scale, g.v_scale,
                        g.upd_full, g.upd_swa, g.active, g.kv)
    ref = []
    for st in (sa, sb):
        o = torch.full_like(g.out, float("nan"))
        call(st, o)
        torch.cuda.synchronize()
        ref.append(o.clone())
    outs = [torch.full_like(g.out, float("nan")) for _ in range(2 * reps)]
    torch.cuda.synchronize()
    for k in range(reps):            # a, b, a, b, ... with nothing in between
        call(sa, outs[2 * k])
        call(sb, outs[2 * k + 1])
    torch.cuda.synchronize()
    assert gk.gk_read_device_error() == 0
    for k in range(reps):
        assert torch.equal(outs[2 * k], ref[0]), ("call a", k)
        assert torch.equal(outs[2 * k + 1], ref[1]), ("call b", k)
