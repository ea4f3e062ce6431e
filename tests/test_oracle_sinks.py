"""Oracle pins for the optional attention sinks (GPT-OSS per-head sink logits;
not on the pages): a sink logit joins the softmax denominator and carries no
value, out = sum_t e^(s_t) v_t / (sum_t e^(s_t) + e^(sink)).

Pinned without re-deriving any score:
  * a sink at -inf (float32 lowest) leaves the output bit-identical;
  * with a sink, every head's output is the sink-free output times one scalar
    alpha_h in (0, 1), the same for all 64 channels;
  * 1/alpha - 1 = e^sink / sum_t e^(s_t), so for two sink values the ratio of
    (1/alpha - 1) is exactly e^(sink1 - sink2);
  * the split-KV combine agrees with the unsplit result with sinks present.
"""
import numpy as np
import pytest

import gk_inputs as gi
import oracle


def _run(name, sinks):
    w = gi.get(name)
    c = gi.make_control(w)
    st = gi.make_step(w, "cpu")
    cache = gi.make_cache(w, c, "cpu")
    sh = oracle.make_shape(**gi.shape_dict(w, c))
    kb = [b[0].numpy().reshape(-1).copy() for b in cache]
    vb = [b[1].numpy().reshape(-1).copy() for b in cache]
    out, s = oracle.decode_attn_stack(sh, gi.bf16_bits(st["q"]), kb, vb, c.k_scale, c.v_scale,
                                      c.cos, c.sin, c.bt_full, c.bt_swa, c.pos, c.pos_w, c.active,
                                      sinks=sinks)
    assert s == 0
    return w, c, out


@pytest.mark.parametrize("name", ["tiny", "gptoss_small"])
def test_minus_infinity_sink_changes_nothing(name):
    w, c, base = _run(name, None)
    _, _, same = _run(name, np.full((w.num_layers, w.num_q_heads), -np.inf, np.float32))
    assert np.array_equal(base, same)


@pytest.mark.parametrize("name", ["tiny", "gptoss_small"])
def test_sink_scales_each_head_and_follows_exp(name):
    w, c, base = _run(name, None)
    rng = np.random.default_rng(3)
    s1 = rng.normal(0.0, 2.0, (w.num_layers, w.num_q_heads)).astype(np.float32)
    s2 = (s1 - 1.5).astype(np.float32)
    _, _, o1 = _run(name, s1)
    _, _, o2 = _run(name, s2)
    act = c.active == 1
    b_ = base[:, act]                     # [NL, rows, Hq, D]
    a1 = (o1[:, act] * b_).sum(-1) / (b_ * b_).sum(-1)   # per-head least-squares scalar
    a2 = (o2[:, act] * b_).sum(-1) / (b_ * b_).sum(-1)
    np.testing.assert_allclose(o1[:, act], a1[..., None] * b_, rtol=0, atol=1e-12)
    np.testing.assert_allclose(o2[:, act], a2[..., None] * b_, rtol=0, atol=1e-12)
    assert (a1 > 0).all() and (a1 < 1).all() and (a2 > a1).all()
    ratio = (1 / a1 - 1) / (1 / a2 - 1)
    d = s1.astype(np.float64) - s2.astype(np.float64)          # ~1.5 after the float32 rounding
    np.testing.assert_allclose(ratio, np.broadcast_to(np.exp(d)[:, None, :], ratio.shape), rtol=1e-9)


def test_split_combine_with_sinks():
    w = gi.get("long_small")
    c = gi.make_control(w)
    st = gi.make_step(w, "cpu")
    cache = gi.make_cache(w, c, "cpu")
    sh = oracle.make_shape(**gi.shape_dict(w, c))
    sinks = np.random.default_rng(5).normal(0, 2, (w.num_layers, w.num_q_heads)).astype(np.float32)
    q = gi.bf16_bits(st["q"])
    args = (q, cache[0][0].numpy().reshape(-1), cache[0][1].numpy().reshape(-1), c.k_scale,
            c.v_scale, c.cos, c.sin, c.bt_full, c.bt_swa, c.pos, c.pos_w, c.active)
    for layer in (0, 1):
        o1, s1 = oracle.attn_one(sh, *args, layer, 0, 0, nsplit=1, sinks=sinks)
        o7, s7 = oracle.attn_one(sh, *args, layer, 0, 0, nsplit=7, sinks=sinks)
        assert s1 == 0 and s7 == 0
        np.testing.assert_allclose(o7, o1, rtol=1e-12, atol=1e-13)
