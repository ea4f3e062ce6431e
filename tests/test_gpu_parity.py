"""GPU parity: the CUDA path (through the C ABI) against the oracle.

Small workloads are compared element by element (every KV byte, every
output).  The five full-size workloads run in the launch configuration the
benchmark times (recommended workspace, persistent grid) and are checked on
every appended KV byte, on untouched cache bytes, on sampled (layer, row, kv
head) outputs recomputed by the oracle, and on properties that hold at any
size.  Tolerances are stated in gk_testlib.
"""
import numpy as np
import pytest
import torch

import gk_inputs as gi
import gk_testlib as tl
import oracle
import paged_fp8_kv_gk_gb300 as gk

pytestmark = pytest.mark.gpu

SMALL = ["tiny", "gptoss_small", "long_small", "ragged_small", "swa_small", "swa_small_sat",
         "swa_small_peaky", "block16_small", "gk120b_rank_small", "block64_small",
         "max_batch", "max_block", "max_layers"]
FULL = ["gptoss_b64", "long_ctx", "ragged_b256", "swa_b512"]


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


# ---------------------------------------------------------------- small workloads
@pytest.mark.parametrize("name", SMALL)
def test_small_step_parity(name):
    w, c, st, cache = _make_cpu(name)
    ref, kb_ref, vb_ref = tl.oracle_step(w, c, st, cache)
    g = tl.GpuStep(w, c, st, cache)
    g.append()
    g.attention()
    torch.cuda.synchronize()
    assert gk.gk_read_device_error() == 0
    for j in range(len(g.cache)):
        assert np.array_equal(g.cache[j][0].cpu().numpy().reshape(-1), kb_ref[j]), ("K", j)
        assert np.array_equal(g.cache[j][1].cpu().numpy().reshape(-1), vb_ref[j]), ("V", j)
    out, of = _f64(g.out), _f64(g.out_f32)
    tl.check_out(out, of, ref, name)
    assert (out[:, c.active == 0] == 0).all() and (of[:, c.active == 0] == 0).all()


@pytest.mark.parametrize("name", ["gptoss_small", "block16_small"])
def test_one_key_rows_return_value_exactly(name):
    """A row whose context is the new token alone returns its dequantised V
    exactly (E4M3 code times a power-of-two scale is a bf16 value)."""
    w, c, st, cache = _make_cpu(name)
    ref, _, _ = tl.oracle_step(w, c, st, cache)
    g = tl.GpuStep(w, c, st, cache)
    g.append()
    g.attention()
    out = _f64(g.out)
    rows = np.nonzero(c.lengths == 1)[0]
    assert rows.size
    assert np.array_equal(out[:, rows], ref[:, rows])


@pytest.mark.parametrize("name", ["long_small", "gptoss_small", "ragged_small"])
def test_split_and_unsplit_agree(name):
    """The recommended workspace lets the planner split long rows (flash-
    decoding partials merged by the combine kernel); the minimum workspace forces
    one unit per row.  Both must meet the tolerance, and the split run must
    actually have split."""
    w, c, st, cache = _make_cpu(name)
    ref, _, _ = tl.oracle_step(w, c, st, cache)
    g = tl.GpuStep(w, c, st, cache)
    g.append()
    g.attention()
    torch.cuda.synchronize()
    hdr = g.workspace[:256].view(torch.int32).cpu().numpy()
    if name == "long_small":
        assert hdr[6] > 0, "expected split-KV partials"     # total split records
    split_out, split_f = _f64(g.out), _f64(g.out_f32)
    ws_min = torch.empty(gk.gk_attn_workspace_min_bytes(g.shape), dtype=torch.uint8, device="cuda")
    g.attention(workspace=ws_min)
    torch.cuda.synchronize()
    hdr2 = ws_min[:256].view(torch.int32).cpu().numpy()
    assert hdr2[6] == 0
    tl.check_out(split_out, split_f, ref, name + "/split")
    tl.check_out(_f64(g.out), _f64(g.out_f32), ref, name + "/unsplit")
    assert gk.gk_read_device_error() == 0


@pytest.mark.parametrize("step", ["split", "fused"])
def test_last_wave_pieces(step):
    """Three long rows over 16 layers: equal chunks would leave a partial last
    wave, so the planner cuts chunks of those rows into pieces that run at the
    end (header word 7 counts them).  Pieces change only where the splits
    fall: every appended KV byte stays bit-exact and sampled outputs meet the
    tolerance, with gk_kv_append + gk_decode_attn_stack and with
    gk_decode_step."""
    w = gi.get("long_cut_small")
    c = gi.make_control(w)
    st = gi.make_step(w, "cuda")
    cache = gi.make_cache(w, c, "cuda")
    pre = [b.clone() for b in cache]
    g = tl.GpuStep(w, c, st, cache)
    if step == "fused":
        g.step()
    else:
        g.append()
        g.attention()
    torch.cuda.synchronize()
    assert gk.gk_read_device_error() == 0
    hdr = g.workspace[:256].view(torch.int32).cpu().numpy()
    assert hdr[7] > 0 and hdr[6] > 0, hdr[:8]
    kc_d, vc_d = tl.device_appended_codes(g)
    kc_o, vc_o = tl.oracle_appended_codes(w, c, st)
    assert np.array_equal(kc_d, kc_o) and np.array_equal(vc_d, vc_o)
    host = {k: gi.bf16_bits(v) for k, v in st.items()}
    G = w.num_q_heads // w.num_kv_heads
    out, of = _f64(g.out), _f64(g.out_f32)
    for b in range(w.batch):
        for j in (0, w.num_layers // 2 - 1):
            res = tl.oracle_row_pair(w, c, host, pre, j, b, kvhs=(0, w.num_kv_heads - 1))
            for (layer, kvh), ref in res.items():
                sl = slice(kvh * G, (kvh + 1) * G)
                tl.check_out(out[layer, b, sl], of[layer, b, sl], ref, f"{step} l{layer} b{b} h{kvh}")


@pytest.mark.parametrize("name,split_len,pieces", [("gptoss_b1_8k", 1024, False),
                                                    ("gptoss_b8_8k", 1024, True)])
def test_plan_choices_at_the_latency_end(name, split_len, pieces):
    """The planner's choices on 36-layer rows of 8192 tokens, on a GPU with
    152 SMs (2432 resident warps): chunks of 1024 tokens (512 would give a row
    16 partials to merge), and chunks cut for the last wave only when the
    chunks make at least one full wave (8 rows: 3.8 waves; 1 row: 0.5).  The
    outputs of sampled rows meet the tolerance."""
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("plan expectations are for 152 SMs")
    w = gi.get(name)
    c = gi.make_control(w)
    st = gi.make_step(w, "cuda")
    cache = gi.make_cache(w, c, "cuda")
    pre = [b.clone() for b in cache]
    g = tl.GpuStep(w, c, st, cache)
    g.append()
    g.attention()
    torch.cuda.synchronize()
    assert gk.gk_read_device_error() == 0
    hdr = g.workspace[:256].view(torch.int32).cpu().numpy()
    assert hdr[4] == split_len and (hdr[7] > 0) == pieces, hdr[:8]
    host = {k: gi.bf16_bits(v) for k, v in st.items()}
    G = w.num_q_heads // w.num_kv_heads
    out, of = _f64(g.out), _f64(g.out_f32)
    for b in sorted({0, w.batch - 1}):
        for j in (0, w.num_layers // 2 - 1):
            res = tl.oracle_row_pair(w, c, host, pre, j, b, kvhs=(0, w.num_kv_heads - 1))
            for (layer, kvh), ref in res.items():
                sl = slice(kvh * G, (kvh + 1) * G)
                tl.check_out(out[layer, b, sl], of[layer, b, sl], ref, f"{name} l{layer} b{b} h{kvh}")


def test_repeat_is_bitwise_deterministic():
    w, c, st, cache = _make_cpu("long_small")
    g = tl.GpuStep(w, c, st, cache)
    g.append()
    g.attention()
    a = g.out.clone()
    af = g.out_f32.clone()
    for _ in range(3):
        g.attention()
        assert torch.equal(g.out, a) and torch.equal(g.out_f32, af)


def test_all_rows_inactive():
    w, c, st, cache = _make_cpu("gptoss_small")
    c.active[:] = 0
    before = [b.clone() for b in cache]
    g = tl.GpuStep(w, c, st, cache)
    g.out.fill_(1.0)
    g.append()
    g.attention()
    torch.cuda.synchronize()
    assert (g.out == 0).all() and (g.out_f32 == 0).all()
    for a, b in zip(g.cache, before):
        assert torch.equal(a.cpu(), b)
    assert gk.gk_read_device_error() == 0


def test_out_f32_optional_gives_same_bf16():
    w, c, st, cache = _make_cpu("gptoss_small")
    g = tl.GpuStep(w, c, st, cache)
    g.append()
    g.attention(out_f32=True)
    a = g.out.clone()
    g.attention(out_f32=False)
    assert torch.equal(a, g.out)


# ---------------------------------------------------------------- device encoder
def test_device_e4m3_encoder_exhaustive():
    """gk_e4m3_quantize with scale 1 over every fp32 pattern with |x| in
    [2^-12, 2^10), both signs, plus random patterns and specials: bit-exact
    with the oracle's encoder."""
    dev = torch.device("cuda")
    mant = torch.arange(1 << 23, dtype=torch.int64, device=dev)
    for e in range(127 - 12, 127 + 10):
        for s in (0, 1):
            bits = ((s << 31) | (e << 23) | mant).to(torch.int64)
            x = (bits - (bits >= 2 ** 31).to(torch.int64) * 2 ** 32).to(torch.int32).view(torch.float32)
            codes = torch.empty(x.numel(), dtype=torch.uint8, device=dev)
            gk.gk_e4m3_quantize(x, 1.0, codes)
            got = codes.cpu().numpy()
            exp = oracle.e4m3_encode(x.cpu().numpy())
            assert np.array_equal(got, exp), (e, s)
    rng = np.random.default_rng(5)
    rb = rng.integers(0, 1 << 32, size=1 << 22, dtype=np.uint64).astype(np.uint32)
    sp = np.array([0, 0x80000000, 0x7F800000, 0xFF800000, 0x7FC00000, 0xFFC00000, 1, 0x80000001,
                   0x00800000, 0x43E00000, 0x43E80000, 0xC3E80000], np.uint32)
    xh = np.concatenate([rb, sp]).view(np.float32)
    x = torch.from_numpy(xh.copy()).to(dev)
    codes = torch.empty(x.numel(), dtype=torch.uint8, device=dev)
    gk.gk_e4m3_quantize(x, 1.0, codes)
    assert np.array_equal(codes.cpu().numpy(), oracle.e4m3_encode(xh))
    # odd length and a non-unit scale (division then encode)
    x = torch.randn(1001, device=dev) * 40
    codes = torch.empty(1001, dtype=torch.uint8, device=dev)
    gk.gk_e4m3_quantize(x, 0.0625, codes)
    xd = x.cpu().numpy()
    assert np.array_equal(codes.cpu().numpy(), oracle.e4m3_encode((xd / np.float32(0.0625)).astype(np.float32)))


# ---------------------------------------------------------------- bounds flags
def test_device_bounds_flags_without_fault():
    """Out-of-range device data is skipped and reported, never dereferenced."""
    w, c, st, cache = _make_cpu("gptoss_small")
    g = tl.GpuStep(w, c, st, cache)
    gk.gk_read_device_error(clear=True)
    # a block id past num_blocks in the full table
    bad = g.bt_full.clone()
    bad[3, 0] = c.num_blocks + 1000
    keep = g.bt_full
    g.bt_full = bad
    g.attention()
    assert gk.gk_read_device_error() & gk.GK_DEVERR_BLOCK
    g.bt_full = keep
    # an update slot past the buffer
    keep = g.upd_full
    g.upd_full = keep.clone()
    g.upd_full[2] = c.num_blocks * w.block_size + 5
    g.append()
    assert gk.gk_read_device_error() & gk.GK_DEVERR_SLOT
    g.upd_full = keep
    # a position beyond the table row
    keep = g.pos
    g.pos = keep.clone()
    g.pos[5] = c.max_blocks_full * w.block_size + 100
    g.attention()
    assert gk.gk_read_device_error() & gk.GK_DEVERR_POS
    g.pos = keep
    g.attention()
    assert gk.gk_read_device_error() == 0


# ---------------------------------------------------------------- full-size workloads
def _kv_untouched(g, pre, c, w):
    """Every cache byte outside the update slots is unchanged."""
    B, Hkv, D = w.block_size, w.num_kv_heads, w.head_dim
    act = torch.as_tensor(np.nonzero(c.active)[0], device=pre[0].device)
    hk = torch.arange(Hkv, device=pre[0].device)
    for j in range(len(pre)):
        a = g.cache[j]
        p = pre[j].clone()
        for i in (2 * j, 2 * j + 1):
            upd = torch.as_tensor((c.upd_swa if i % 2 == 0 else c.upd_full).astype(np.int64),
                                  device=p.device)[act]
            pb, t = upd // B, upd % B
            kv_p = p[0].view(c.num_blocks, Hkv, B // 2, D, 2)
            kv_a = a[0].view(c.num_blocks, Hkv, B // 2, D, 2)
            ix = (pb[:, None], hk[None, :], (t // 2)[:, None], slice(None), (t % 2)[:, None])
            kv_p[ix] = kv_a[ix]
            iv = (pb[:, None], hk[None, :], t[:, None], slice(None))
            p[1][iv] = a[1][iv]
        assert torch.equal(p, a), ("cache bytes outside the update slots changed", j)
        del p


@pytest.mark.parametrize("name", FULL)
def test_full_size_parity(name):
    """A full-size workload in the benchmark's launch configuration
    (recommended workspace, persistent grid): every appended KV byte
    bit-exact, every other cache byte unchanged, and every output element of
    every (layer, row, q head) against the oracle, the whole output computed
    by the oracle row by row on the host cores."""
    w = gi.get(name)
    c = gi.make_control(w)
    st = gi.make_step(w, "cuda")
    cache = gi.make_cache(w, c, "cuda")
    pre = [b.clone() for b in cache]
    g = tl.GpuStep(w, c, st, cache)
    g.append()
    g.attention()
    torch.cuda.synchronize()
    assert gk.gk_read_device_error() == 0

    # every appended byte, bit-exact
    kc_d, vc_d = tl.device_appended_codes(g)
    kc_o, vc_o = tl.oracle_appended_codes(w, c, st)
    act = c.active == 1
    assert np.array_equal(kc_d[:, act], kc_o[:, act])
    assert np.array_equal(vc_d[:, act], vc_o[:, act])
    _kv_untouched(g, pre, c, w)

    # the whole output against the oracle
    out = g.out.float().cpu().numpy().astype(np.float64)
    of = g.out_f32.cpu().numpy().astype(np.float64)
    del g, cache
    host = {k: gi.bf16_bits(v) for k, v in st.items()}
    ref = tl.oracle_full_output(w, c, host, pre)
    assert (out[:, ~act] == 0).all() and (of[:, ~act] == 0).all()
    stats = tl.check_out(out, of, ref, f"{name} whole output")
    print(f"{name}: {stats['elements']} elements compared, {stats['bf16_widened']} bf16 elements "
          f"within one bf16 step but beyond {tl.MAX_ABS}")


def test_full_size_repeat_bitwise():
    """Split merges happen in split order whatever the arrival order: repeated
    full-size calls give bit-identical outputs (and no device error)."""
    w = gi.get("gptoss_b64")
    c = gi.make_control(w)
    st = gi.make_step(w, "cuda")
    cache = gi.make_cache(w, c, "cuda")
    g = tl.GpuStep(w, c, st, cache)
    g.append()
    g.attention()
    torch.cuda.synchronize()
    ref, refb = g.out_f32.clone(), g.out.clone()
    for _ in range(20):
        g.attention()
        torch.cuda.synchronize()
        assert torch.equal(g.out_f32, ref) and torch.equal(g.out, refb)
    assert gk.gk_read_device_error() == 0


@pytest.mark.parametrize("case", ["q_zero", "v_zero", "k_zero"])
def test_degenerate_inputs(case):
    """q = 0 (every score 0: the normaliser's all-zero branch; the output is
    the mean of the values), V = 0 (output exactly 0), K = 0 (uniform weights)
    -- against the oracle on the same inputs."""
    w, c, st, cache = _make_cpu("gptoss_small")
    st = {k: v.clone() for k, v in st.items()}
    cache = [b.clone() for b in cache]
    if case == "q_zero":
        st["q"].zero_()
    elif case == "v_zero":
        st["v_new"].zero_()
        for b in cache:
            b[1].zero_()
    else:
        st["k_new"].zero_()
        for b in cache:
            b[0].zero_()
    ref, _, _ = tl.oracle_step(w, c, st, cache)
    g = tl.GpuStep(w, c, st, cache)
    g.append()
    g.attention()
    torch.cuda.synchronize()
    assert gk.gk_read_device_error() == 0
    out, of = _f64(g.out), _f64(g.out_f32)
    tl.check_out(out, of, ref, case)
    if case == "v_zero":
        assert (g.out_f32 == 0).all()
