"""Pins for the oracle's append and attention (CPU only).

The oracle is checked against: an independent numpy/torch restatement that
reads K through torch's .view() of the page's packed shape, decodes codes with
torch's float8 cast and rotates q by complex multiplication; contiguous-cache
attention (paged == contiguous, window layer == last-W keys); closed-form
special cases (one key returns V exactly, equal keys return the mean, a
dominant logit returns its value); split invariance of the combine; and the
library float8 cast for the append path.
"""
import numpy as np
import pytest
import torch

import gk_inputs as gi
import oracle

# ------------------------------------------------------------------ helpers


def _setup(name):
    w = gi.get(name)
    c = gi.make_control(w)
    st = gi.make_step(w, "cpu")
    cache = gi.make_cache(w, c, "cpu")
    return w, c, st, cache


def _np_bufs(cache):
    k = [b[0].contiguous().numpy().reshape(-1) for b in cache]
    v = [b[1].contiguous().numpy().reshape(-1) for b in cache]
    return k, v


def _shape(w, c):
    return oracle.make_shape(**gi.shape_dict(w, c))


def _brute_step(w, c, q_bits, cache):
    """Independent restatement of the whole decode-attention step in numpy."""
    NL, Bt, Hq, Hkv, D, B, W = (w.num_layers, w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                w.block_size, w.window)
    G = Hq // Hkv
    out = np.zeros((NL, Bt, Hq, D))
    qf = torch.from_numpy(q_bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    for i in range(NL):
        buf = cache[i // 2]
        kview = buf[0].view(c.num_blocks, Hkv, B // 2, D, 2)      # the page's packed view
        vview = buf[1]                                           # [nb, Hkv, B, D]
        for b in range(Bt):
            if not c.active[b]:
                continue
            pos = int(c.pos[b])
            if i % 2 == 0:   # sliding window: absolute keys, mapped into the trimmed frame
                shift = pos - int(c.pos_w[b])
                keys = np.arange(max(0, pos - W + 1), pos + 1)
                frame = keys - shift
                row = c.bt_swa[b]
            else:
                keys = np.arange(0, pos + 1)
                frame = keys
                row = c.bt_full[b]
            pbs = torch.as_tensor(row[frame // B].astype(np.int64))
            offs = torch.as_tensor(frame % B)
            for kvh in range(Hkv):
                kc = kview[pbs, kvh, offs // 2, :, offs % 2]         # [n, D] codes
                vc = vview[pbs, kvh, offs, :]
                kd = kc.contiguous().view(torch.float8_e4m3fn).to(torch.float64).numpy() * float(c.k_scale[i])
                vd = vc.contiguous().view(torch.float8_e4m3fn).to(torch.float64).numpy() * float(c.v_scale[i])
                for g in range(G):
                    h = kvh * G + g
                    x = qf[i, b, h]
                    rot = (x[:D // 2] + 1j * x[D // 2:]) * (
                        c.cos[b].astype(np.float64) + 1j * c.sin[b].astype(np.float64))
                    qr = np.concatenate([rot.real, rot.imag])
                    s = kd @ qr / np.sqrt(D)
                    p = np.exp(s - s.max())
                    out[i, b, h] = (p[:, None] * vd).sum(0) / p.sum()
    return out


# ------------------------------------------------------------------ whole step
@pytest.mark.parametrize("name", ["tiny", "block16_small", "gptoss_small", "swa_small",
                                  "gk120b_rank_small", "block64_small"])
def test_oracle_step_matches_independent_restatement(name):
    w, c, st, cache = _setup(name)
    q = gi.bf16_bits(st["q"])
    kb, vb = _np_bufs(cache)
    out, status = oracle.decode_attn_stack(_shape(w, c), q, kb, vb, c.k_scale, c.v_scale, c.cos, c.sin,
                                           c.bt_full, c.bt_swa, c.pos, c.pos_w, c.active)
    assert status == 0
    ref = _brute_step(w, c, q, cache)
    assert np.max(np.abs(out - ref)) < 1e-11


@pytest.mark.parametrize("name", ["gptoss_small", "ragged_small", "block16_small"])
def test_each_row_equals_that_row_alone(name):
    """Rows of a batch are independent problems: the whole-step result for
    row b equals (bit for bit) the step run on a batch holding row b alone
    (its q, cos/sin, table rows, positions and activity, the same caches)."""
    w, c, st, cache = _setup(name)
    q = gi.bf16_bits(st["q"])
    kb, vb = _np_bufs(cache)
    args = lambda rows: (q[:, rows], kb, vb, c.k_scale, c.v_scale, c.cos[rows], c.sin[rows],  # noqa: E731
                         c.bt_full[rows], c.bt_swa[rows], c.pos[rows], c.pos_w[rows], c.active[rows])
    full, status = oracle.decode_attn_stack(_shape(w, c), *args(slice(None)))
    assert status == 0
    d = gi.shape_dict(w, c)
    d["batch"] = 1
    sh1 = oracle.make_shape(**d)
    for b in range(w.batch):
        one, status = oracle.decode_attn_stack(sh1, *args(slice(b, b + 1)))
        assert status == 0
        assert np.array_equal(one[:, 0], full[:, b]), (name, b)


@pytest.mark.parametrize("name", ["gptoss_small", "max_layers"])
def test_layer_reads_group_buffer_i_over_2(name):
    """Layer i reads group buffer i // 2 with its own V scale ("Kernel
    contract"): fill every V byte of group buffer j with the code of 2^(j % 4)
    and the output of every active (layer, row, head) is exactly
    2^((i // 2) % 4) * v_scale[i], whatever the keys (constant values)."""
    w, c, st, cache = _setup(name)
    q = gi.bf16_bits(st["q"])
    kb, vb = _np_bufs(cache)
    vb = [np.full_like(v, 0x38 + 8 * (j % 4)) for j, v in enumerate(vb)]   # 1, 2, 4, 8
    out, status = oracle.decode_attn_stack(_shape(w, c), q, kb, vb, c.k_scale, c.v_scale, c.cos,
                                           c.sin, c.bt_full, c.bt_swa, c.pos, c.pos_w, c.active)
    assert status == 0
    for i in range(w.num_layers):
        want = 2.0 ** ((i // 2) % 4) * float(c.v_scale[i])
        assert (out[i, c.active == 1] == want).all(), (name, i)


@pytest.mark.parametrize("name", ["gptoss_small", "block16_small"])
def test_step_is_per_unit_attention_on_group_buffer_i_over_2(name):
    """The whole-step routine is the per-(layer, row, kv head) attention (whose
    arithmetic the closed-form and contiguous-cache pins fix) applied with
    group buffer i // 2 ("Kernel contract"), its output placed at heads
    kvh*G .. kvh*G + G - 1 of row b, layer i."""
    w, c, st, cache = _setup(name)
    q = gi.bf16_bits(st["q"])
    kb, vb = _np_bufs(cache)
    sh = _shape(w, c)
    out, status = oracle.decode_attn_stack(sh, q, kb, vb, c.k_scale, c.v_scale, c.cos, c.sin,
                                           c.bt_full, c.bt_swa, c.pos, c.pos_w, c.active)
    assert status == 0
    G = w.num_q_heads // w.num_kv_heads
    for i in range(w.num_layers):
        for b in range(w.batch):
            for kvh in range(w.num_kv_heads):
                one, status = oracle.attn_one(sh, q, kb[i // 2], vb[i // 2], c.k_scale, c.v_scale,
                                              c.cos, c.sin, c.bt_full, c.bt_swa, c.pos, c.pos_w,
                                              c.active, i, b, kvh)
                assert status == 0
                assert np.array_equal(out[i, b, kvh * G:(kvh + 1) * G], one), (i, b, kvh)


def test_inactive_rows_are_zero():
    w, c, st, cache = _setup("ragged_small")
    assert (c.active == 0).any()
    kb, vb = _np_bufs(cache)
    out, _ = oracle.decode_attn_stack(_shape(w, c), gi.bf16_bits(st["q"]), kb, vb, c.k_scale,
                                      c.v_scale, c.cos, c.sin, c.bt_full, c.bt_swa, c.pos, c.pos_w,
                                      c.active)
    assert (out[:, c.active == 0] == 0).all()
    assert (np.abs(out[:, c.active == 1]).sum(-1) > 0).all()


# ------------------------------------------------------------------ P6 / P7
def _window_case(L, B=16, W=128, Hkv=2, G=4, D=64, seed=0, identity=False):
    """One sequence; layer 0 (sliding window) reads the trimmed table, layer 1
    (full) the full table.  Both layers' key/value rows come from one
    contiguous array of L positions, placed into the pool by the tables."""
    rng = np.random.default_rng(seed)
    nfull = -(-L // B)
    b0 = max(0, L - W) // B
    nswa = (L - 1) // B - b0 + 1
    nb = nfull + nswa + 1
    perm = rng.permutation(nb - 1)
    if identity:
        perm = np.arange(nb - 1)
    full_ids, swa_ids = perm[:nfull], perm[nfull:nfull + nswa]
    mbs = -(-(W + B - 1) // B)
    bt_full = np.full((1, nfull), nb - 1, np.int32)
    bt_full[0] = full_ids
    bt_swa = np.full((1, mbs), nb - 1, np.int32)
    bt_swa[0, :nswa] = swa_ids
    kc = rng.integers(0, 0x7F, size=(L, Hkv, D)).astype(np.uint8) | (
        rng.integers(0, 2, size=(L, Hkv, D)).astype(np.uint8) << 7)
    kc[kc == 0x7F] = 0x7E
    kc[kc == 0xFF] = 0xFE
    vc = rng.integers(0, 0x78, size=(L, Hkv, D)).astype(np.uint8)
    kbuf = np.zeros(nb * Hkv * B * D, np.uint8)
    vbuf = np.zeros(nb * Hkv * B * D, np.uint8)
    for a in range(L):           # place every position for the full layer
        pb = full_ids[a // B]
        for h in range(Hkv):
            for e in range(D):
                kbuf[oracle.k_offset(Hkv, B, D, pb, h, a % B, e)] = kc[a, h, e]
                vbuf[oracle.v_offset(Hkv, B, D, pb, h, a % B, e)] = vc[a, h, e]
    for a in range(b0 * B, L):   # and the window blocks for the sliding-window layer
        pb = swa_ids[a // B - b0]
        for h in range(Hkv):
            for e in range(D):
                kbuf[oracle.k_offset(Hkv, B, D, pb, h, a % B, e)] = kc[a, h, e]
                vbuf[oracle.v_offset(Hkv, B, D, pb, h, a % B, e)] = vc[a, h, e]
    sh = oracle.make_shape(num_layers=2, batch=1, num_q_heads=Hkv * G, num_kv_heads=Hkv, head_dim=D,
                           block_size=B, num_blocks=nb, window=W, max_blocks_full=nfull,
                           max_blocks_swa=mbs)
    q = torch.randn(2, 1, Hkv * G, D, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)
    ang = rng.uniform(-3, 3, D // 2)
    cos = np.cos(ang).astype(np.float32)[None]
    sin = np.sin(ang).astype(np.float32)[None]
    scales = np.array([1 / 16, 1 / 32], np.float32)
    ctl = dict(bt_full=bt_full, bt_swa=bt_swa, pos=np.array([L - 1], np.int32),
               pos_w=np.array([L - 1 - b0 * B], np.int32), active=np.ones(1, np.uint8))
    return sh, gi.bf16_bits(q), kbuf, vbuf, scales, cos, sin, ctl, kc, vc


def _contig_attention(q_bits, kc, vc, ks, vs, cos, sin, keys, kvh, G, D):
    qf = torch.from_numpy(q_bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    kd = oracle.e4m3_decode(kc[keys, kvh]) * ks
    vd = oracle.e4m3_decode(vc[keys, kvh]) * vs
    res = []
    for g in range(G):
        x = qf[kvh * G + g]
        z = (x[:D // 2] + 1j * x[D // 2:]) * (cos[0].astype(np.float64) + 1j * sin[0].astype(np.float64))
        s = kd @ np.concatenate([z.real, z.imag]) / np.sqrt(D)
        p = np.exp(s - s.max())
        res.append((p[:, None] * vd).sum(0) / p.sum())
    return np.array(res)


WINDOW_LENGTHS = [1, 2, 15, 16, 17, 127, 128, 129, 130, 143, 144, 145, 159, 160, 161, 175, 191, 300]


@pytest.mark.parametrize("L", WINDOW_LENGTHS)
def test_window_layer_equals_last_W_keys_of_contiguous_cache(L):
    """P6: layer 0 through the trimmed table and window-frame position equals
    attention over the last W positions of the contiguous cache; layer 1
    through the full table equals attention over all L positions.  Lengths
    cover L % B == B - 1 and the window start at several block offsets.  K and
    V carry different scales."""
    B, W, G, D = 16, 128, 4, 64
    sh, q, kbuf, vbuf, sc, cos, sin, ctl, kc, vc = _window_case(L, B=B, W=W, G=G, seed=L)
    sv = np.array([1 / 4, 1 / 128], np.float32)
    for layer, keys in ((0, np.arange(max(0, L - W), L)), (1, np.arange(L))):
        for kvh in range(2):
            out, st = oracle.attn_one(sh, q, kbuf, vbuf, sc, sv, cos, sin, ctl["bt_full"],
                                      ctl["bt_swa"], ctl["pos"], ctl["pos_w"], ctl["active"],
                                      layer, 0, kvh)
            assert st == 0
            ref = _contig_attention(q[layer, 0], kc, vc, sc[layer], sv[layer], cos, sin, keys, kvh, G, D)
            assert np.max(np.abs(out - ref)) < 1e-11, (L, layer, kvh)


@pytest.mark.parametrize("L", [1, 37, 160, 300])
def test_paged_equals_contiguous(L):
    """P7: a random-permutation table gives bit-identical results to the
    identity table over the same positions."""
    outs = []
    for ident in (False, True):
        sh, q, kbuf, vbuf, sc, cos, sin, ctl, kc, vc = _window_case(L, seed=99, identity=ident)
        res = []
        for layer in (0, 1):
            for kvh in range(2):
                o, st = oracle.attn_one(sh, q, kbuf, vbuf, sc, sc, cos, sin, ctl["bt_full"],
                                        ctl["bt_swa"], ctl["pos"], ctl["pos_w"], ctl["active"],
                                        layer, 0, kvh)
                assert st == 0
                res.append(o)
        outs.append(np.array(res))
    assert np.array_equal(outs[0], outs[1])


# ------------------------------------------------------------------ P8 special cases
def test_one_key_returns_value_exactly():
    sh, q, kbuf, vbuf, sc, cos, sin, ctl, kc, vc = _window_case(1, seed=3)
    for layer in (0, 1):
        for kvh in range(2):
            o, _ = oracle.attn_one(sh, q, kbuf, vbuf, sc, sc, cos, sin, ctl["bt_full"], ctl["bt_swa"],
                                   ctl["pos"], ctl["pos_w"], ctl["active"], layer, 0, kvh)
            v = oracle.e4m3_decode(vc[0, kvh]) * sc[layer]
            assert np.array_equal(o, np.broadcast_to(v, o.shape))


def test_equal_keys_return_mean_and_dominant_logit_returns_its_value():
    L = 200
    sh, q, kbuf, vbuf, sc, cos, sin, ctl, kc, vc = _window_case(L, seed=4)
    B, Hkv, D = 16, 2, 64
    # equal keys: overwrite every K code with one row
    k2 = kbuf.copy()
    row = kc[0, 0]
    for pb in range(sh.num_blocks):
        for h in range(Hkv):
            for t in range(B):
                for e in range(D):
                    k2[oracle.k_offset(Hkv, B, D, pb, h, t, e)] = row[e]
    o, _ = oracle.attn_one(sh, q, k2, vbuf, sc, sc, cos, sin, ctl["bt_full"], ctl["bt_swa"], ctl["pos"],
                           ctl["pos_w"], ctl["active"], 1, 0, 0)
    mean = (oracle.e4m3_decode(vc[:, 0]) * sc[1]).mean(0)
    assert np.max(np.abs(o - mean)) < 1e-12
    # dominant logit: q . k huge for one key (k = +-448 aligned with q's sign), others zero
    k3 = np.zeros_like(kbuf)
    qf = torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()[1, 0, 0]
    z = (qf[:32] + 1j * qf[32:]) * (cos[0].astype(np.float64) + 1j * sin[0].astype(np.float64))
    qr = np.concatenate([z.real, z.imag])
    star = 77
    pb = ctl["bt_full"][0, star // B]
    for e in range(D):
        k3[oracle.k_offset(Hkv, B, D, pb, 0, star % B, e)] = 0x7E if qr[e] > 0 else 0xFE
    o, _ = oracle.attn_one(sh, q, k3, vbuf, np.array([1.0, 1.0], np.float32), sc, cos, sin,
                           ctl["bt_full"], ctl["bt_swa"], ctl["pos"], ctl["pos_w"], ctl["active"], 1, 0, 0)
    v_star = oracle.e4m3_decode(vc[star, 0]) * sc[1]
    assert np.max(np.abs(o[0] - v_star)) < 1e-9


def test_gqa_head_to_kv_head_map():
    """q head h reads kv head h // G: give each kv head a constant V row."""
    L, B, Hkv, G, D = 50, 16, 2, 4, 64
    sh, q, kbuf, vbuf, sc, cos, sin, ctl, kc, vc = _window_case(L, seed=8)
    v2 = vbuf.copy()
    consts = {0: 0x38, 1: 0x40}   # 1.0 and 2.0
    for pb in range(sh.num_blocks):
        for h in range(Hkv):
            for t in range(B):
                for e in range(D):
                    v2[oracle.v_offset(Hkv, B, D, pb, h, t, e)] = consts[h]
    for kvh in range(Hkv):
        o, _ = oracle.attn_one(sh, q, kbuf, v2, sc, np.ones(2, np.float32), cos, sin, ctl["bt_full"],
                               ctl["bt_swa"], ctl["pos"], ctl["pos_w"], ctl["active"], 1, 0, kvh)
        assert np.allclose(o, 1.0 + kvh, atol=1e-14)


# ------------------------------------------------------------------ P9 split combine
@pytest.mark.parametrize("nsplit", [2, 7, 64, 10000])
def test_split_combine_invariance(nsplit):
    sh, q, kbuf, vbuf, sc, cos, sin, ctl, kc, vc = _window_case(300, seed=11)
    args = (sh, q, kbuf, vbuf, sc, sc, cos, sin, ctl["bt_full"], ctl["bt_swa"], ctl["pos"],
            ctl["pos_w"], ctl["active"])
    for layer in (0, 1):
        ref, _ = oracle.attn_one(*args, layer, 0, 1, 1)
        got, _ = oracle.attn_one(*args, layer, 0, 1, nsplit)
        assert np.max(np.abs(got - ref)) < 1e-12


# ------------------------------------------------------------------ append pins
def _append(w, c, st, cache):
    kb, vb = _np_bufs(cache)
    kb = [a.copy() for a in kb]
    vb = [a.copy() for a in vb]
    status = oracle.kv_append(_shape(w, c), gi.bf16_bits(st["k_new"]), gi.bf16_bits(st["v_new"]),
                              c.cos, c.sin, c.k_scale, c.v_scale, c.upd_full, c.upd_swa, c.active,
                              kb, vb)
    return kb, vb, status


@pytest.mark.parametrize("name", ["tiny", "ragged_small", "block16_small"])
def test_append_touches_exactly_the_update_slots(name):
    w, c, st, cache = _setup(name)
    kb0, vb0 = _np_bufs(cache)
    kb, vb, status = _append(w, c, st, cache)
    assert status == 0
    B, Hkv, D = w.block_size, w.num_kv_heads, w.head_dim
    for j in range(w.num_layers // 2):
        allowed_k = np.zeros(kb0[j].size, bool)
        allowed_v = np.zeros(vb0[j].size, bool)
        for i in (2 * j, 2 * j + 1):
            upd = c.upd_swa if i % 2 == 0 else c.upd_full
            for b in range(w.batch):
                if not c.active[b]:
                    continue
                pb, t = divmod(int(upd[b]), B)
                for h in range(Hkv):
                    for e in range(D):
                        allowed_k[oracle.k_offset(Hkv, B, D, pb, h, t, e)] = True
                        allowed_v[oracle.v_offset(Hkv, B, D, pb, h, t, e)] = True
        assert not (kb[j] != kb0[j])[~allowed_k].any()
        assert not (vb[j] != vb0[j])[~allowed_v].any()


def test_append_codes_match_library_cast_and_values():
    """Read back through the page's packed view: V codes equal torch's float8
    cast of v / scale; decoded K values are within half an E4M3 step of the
    exact rotation of k / scale, and values past 448 saturate.  The V scales
    are set apart from the K scales (the workload uses one scale for both),
    so that each half is checked against its own scale."""
    w, c, st, cache = _setup("swa_small_sat")
    c.v_scale = np.array([2.0 ** -(2 + i % 4) for i in range(w.num_layers)], np.float32)
    assert not np.array_equal(c.v_scale, c.k_scale)
    kb, vb, _ = _append(w, c, st, cache)
    B, Hkv, D = w.block_size, w.num_kv_heads, w.head_dim
    kf = st["k_new"].to(torch.float64).numpy()
    vf = st["v_new"].to(torch.float32)
    sat = 0
    for i in range(w.num_layers):
        j = i // 2
        kview = torch.from_numpy(kb[j]).view(c.num_blocks, Hkv, B // 2, D, 2)
        vview = torch.from_numpy(vb[j]).view(c.num_blocks, Hkv, B, D)
        upd = c.upd_swa if i % 2 == 0 else c.upd_full
        for b in range(w.batch):
            pb, t = divmod(int(upd[b]), B)
            kcodes = kview[pb, :, t // 2, :, t % 2].numpy()          # [Hkv, D]
            vcodes = vview[pb, :, t, :].numpy()
            vexp = (vf[i, b] / float(c.v_scale[i])).clamp(-448, 448).to(torch.float8_e4m3fn)
            assert np.array_equal(vcodes, vexp.view(torch.uint8).numpy())
            kx = kf[i, b]
            z = (kx[:, :32] + 1j * kx[:, 32:]) * (c.cos[b].astype(np.float64) + 1j * c.sin[b].astype(np.float64))
            exact = np.concatenate([z.real, z.imag], axis=1) / float(c.k_scale[i])
            dec = oracle.e4m3_decode(kcodes)
            big = np.abs(exact) > 448
            sat += int(big.sum())
            assert np.array_equal(dec[big], np.sign(exact[big]) * 448)
            small = ~big & (np.abs(exact) >= 2 ** -6)
            rel = np.abs(dec[small] - exact[small]) / np.abs(exact[small])
            assert rel.max() <= 2 ** -4 * (1 + 1e-5)
            sub = ~big & ~small
            assert np.abs(dec[sub] - exact[sub]).max(initial=0) <= 2 ** -10 * (1 + 1e-5)
    assert sat > 0   # the probe saturates


def test_append_inactive_rows_write_nothing():
    w, c, st, cache = _setup("ragged_small")
    act0 = c.active.copy()
    c.active[:] = 0
    kb0, vb0 = _np_bufs(cache)
    kb, vb, _ = _append(w, c, st, cache)
    c.active[:] = act0
    for j in range(len(kb)):
        assert np.array_equal(kb[j], kb0[j]) and np.array_equal(vb[j], vb0[j])
