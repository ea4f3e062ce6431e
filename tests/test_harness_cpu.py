"""CPU checks of the test harness itself: the compact-pool helpers used for the
full-size sampled parity checks give exactly what the whole-step oracle gives."""
import numpy as np
import pytest

import gk_inputs as gi
import gk_testlib as tl


@pytest.mark.parametrize("name", ["tiny", "ragged_small", "block16_small"])
def test_row_pair_sampler_equals_whole_step(name):
    w = gi.get(name)
    c = gi.make_control(w)
    st = gi.make_step(w, "cpu")
    cache = gi.make_cache(w, c, "cpu")
    full, _, _ = tl.oracle_step(w, c, st, cache)
    host = {k: gi.bf16_bits(v) for k, v in st.items()}
    G = w.num_q_heads // w.num_kv_heads
    for b in range(w.batch):
        if not c.active[b]:
            continue
        for j in range(w.num_layers // 2):
            res = tl.oracle_row_pair(w, c, host, cache, j, b)
            for (layer, kvh), o in res.items():
                assert np.array_equal(o, full[layer, b, kvh * G:(kvh + 1) * G]), (b, layer, kvh)


@pytest.mark.parametrize("name", ["tiny", "ragged_small", "swa_small", "gk120b_rank_small"])
def test_threaded_whole_output_equals_whole_step(name):
    """The whole-output oracle used at full size (rows on host threads, blocks
    copied one layer pair at a time) gives exactly the whole-step oracle's
    output, zeros on inactive rows included."""
    w = gi.get(name)
    c = gi.make_control(w)
    st = gi.make_step(w, "cpu")
    cache = gi.make_cache(w, c, "cpu")
    full, _, _ = tl.oracle_step(w, c, st, cache)
    host = {k: gi.bf16_bits(v) for k, v in st.items()}
    got = tl.oracle_full_output(w, c, host, cache, threads=3)
    assert np.array_equal(got, full)


@pytest.mark.parametrize("name", ["tiny", "ragged_small", "swa_small_sat"])
def test_appended_codes_helper_equals_whole_buffer_append(name):
    w = gi.get(name)
    c = gi.make_control(w)
    st = gi.make_step(w, "cpu")
    cache = gi.make_cache(w, c, "cpu")
    _, kb, vb = tl.oracle_step(w, c, st, cache)
    kc, vc = tl.oracle_appended_codes(w, c, st)
    B, Hkv, D = w.block_size, w.num_kv_heads, w.head_dim
    for i in range(w.num_layers):
        upd = c.upd_swa if i % 2 == 0 else c.upd_full
        kview = kb[i // 2].reshape(c.num_blocks, Hkv, B // 2, D, 2)
        vview = vb[i // 2].reshape(c.num_blocks, Hkv, B, D)
        for b in range(w.batch):
            if not c.active[b]:
                continue
            pb, t = divmod(int(upd[b]), B)
            assert np.array_equal(kc[i, b], kview[pb, :, t // 2, :, t % 2])
            assert np.array_equal(vc[i, b], vview[pb, :, t, :])


def _launch_list(path, launches):
    hdr = '"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream",' \
          '"Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit",' \
          '"Metric Value"\n'
    rows = []
    for i, (k, rd, wr, t) in enumerate(launches):
        for m, v in (("dram__bytes_read.sum", rd), ("dram__bytes_write.sum", wr),
                     ("gpu__time_duration.sum", t)):
            rows.append(f'"{i}","1","python","h","{k}","1","7","(128, 1, 1)","(608, 1, 1)","0",'
                        f'"10.3","Command line profiler metrics","{m}","byte","{v:,}"\n')
    path.write_text(hdr + "".join(rows))


def test_bench_records_traffic_from_an_ncu_launch_list(tmp_path, monkeypatch):
    """bench.py --record-traffic: the attention kernel's launches of a reduced
    case are averaged (other kernels ignored), stamped with the current source
    hash and the case's algorithmic bytes; the full workload's traffic is that
    figure scaled by the ratio of algorithmic bytes."""
    import json
    import bench
    csv_path = tmp_path / "launches.csv"
    _launch_list(csv_path, [("void attn_kernel<1, 1>(AttnParams)", 100, 10, 5),
                            ("plan_kernel(PlanParams)", 7, 0, 1),
                            ("void attn_kernel<1, 1>(AttnParams)", 300, 30, 7)])
    out = tmp_path / "traffic.json"
    e = bench.record_traffic("gptoss_b16", str(csv_path), str(out))
    assert e["dram_read_bytes"] == 200 and e["dram_write_bytes"] == 20
    assert e["dram_bytes_per_launch"] == 220 and e["launches_averaged"] == 2
    assert e["kernel_src_sha"] == bench.attn_source_hash()
    small = gi.get("gptoss_b16")
    assert e["alg_bytes_per_launch"] == bench.alg_bytes(small, gi.make_control(small))
    assert "-k regex:attn_kernel" in e["command"] and "-c 3" in e["command"]
    assert json.loads(out.read_text())["gptoss_b16"]["dram_bytes_per_launch"] == 220
    # the full workload reads its traffic from the reduced case, scaled
    profiles = tmp_path / "profiles"
    profiles.mkdir()
    (profiles / "attn_traffic.json").write_text(out.read_text())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "attn_source_hash", lambda: e["kernel_src_sha"])
    full = gi.get("gptoss_b64")
    cf = gi.make_control(full)
    got, case, scale = bench.recorded_traffic(full, cf)
    assert case == "gptoss_b16"
    assert scale == pytest.approx(bench.alg_bytes(full, cf) / e["alg_bytes_per_launch"])
    assert got == round(220 * scale)
    # a capture taken on another kernel source is not used
    monkeypatch.setattr(bench, "attn_source_hash", lambda: "0" * 16)
    assert bench.recorded_traffic(full, cf) is None


def test_check_out_counts_the_one_step_allowance():
    """The bf16 bar: 1.5e-2 absolute, widened to one bf16 step where that step
    is larger (|x| >= 4, step 2^-5); every widened element is counted and
    listed in the session's report."""
    import oracle
    ref = oracle.round_bf16(np.linspace(-8.0, 8.0, 1001))
    out = ref.copy()
    big = np.flatnonzero(np.abs(ref) >= 4.0)[:3]
    small = np.flatnonzero(np.abs(ref) < 1.0)[0]
    out[big] += np.array([0.02, 0.025, 0.03])   # beyond 1.5e-2, within one step
    out[small] += 0.01                          # within 1.5e-2
    n0 = len(tl.REPORT)
    st = tl.check_out(out, None, ref, "allowance probe")
    assert st["bf16_widened"] == 3 and st["elements"] == ref.size
    assert tl.REPORT[n0:] == [("allowance probe", st)]
    out[small] += 0.01                          # 0.02 where the step is 2^-8: too far
    with pytest.raises(AssertionError):
        tl.check_out(out, None, ref, "too far")
