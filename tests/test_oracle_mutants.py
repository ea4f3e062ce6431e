"""Mutation check of the oracle's pins (CPU only; opt-in, about an hour).

Each case plants one plausible mistake in a copy of oracle/gk_oracle.c (a
wrong constant, sign, index or scale; a dropped term or guard; a transposed
operand or layout; a swapped table or update index), builds that copy and runs
the oracle's pin tests against it.  A case passes when at least one pin fails
on the mutant.  The independent numpy restatement of the whole step is left
out of the pins run here, so that what catches each mistake is a check fixed
by the pages or by the mathematics: the OCP E4M3 table and brute-force
rounding, torch's float8 cast, closed forms of attention (one key, equal keys,
a dominant logit, constant values per kv head), contiguous-cache and
last-W-keys equivalences, split invariance, RoPE identities, the DI block
rule by brute force and the page's region and landing definitions.

Runs only with GK_ORACLE_MUTANTS=1 (each case rebuilds the oracle and runs
the pins, stopping at the first failure).  The unmutated copy must pass.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = open(os.path.join(ROOT, "oracle", "gk_oracle.c")).read()
PIN_TESTS = ["tests/test_oracle_codec_layout.py", "tests/test_oracle_attention.py",
             "tests/test_oracle_kv_forms.py", "tests/test_oracle_sinks.py",
             "tests/test_di_landing_cpu.py"]
NOT_PINS = "not independent_restatement"

pytestmark = pytest.mark.skipif(os.environ.get("GK_ORACLE_MUTANTS") != "1",
                                reason="opt-in: GK_ORACLE_MUTANTS=1 (about an hour of CPU)")

MUTANTS = [
 ("decode_bias", "ldexp(1.0 + (double)m / 8.0, ef - 7)", "ldexp(1.0 + (double)m / 8.0, ef - 8)"),
 ("decode_mant", "(double)m / 8.0", "(double)m / 16.0"),
 ("decode_sub", "ldexp((double)m, -9)", "ldexp((double)m, -10)"),
 ("decode_nan", "if (ef == 15 && m == 7)", "if (ef == 15 && m == 8)"),
 ("decode_sign", "return s ? -v : v;", "return v;"),
 ("encode_sat", "return (uint8_t)(sign | 0x7E);", "return (uint8_t)(sign | 0x7F);"),
 ("encode_floor", "n = nearbyint(ldexp(a, 3 - (e2 - 1)));", "n = floor(ldexp(a, 3 - (e2 - 1)));"),
 ("encode_ties_away", "n = nearbyint(ldexp(a, 3 - (e2 - 1)));", "n = round(ldexp(a, 3 - (e2 - 1)));"),
 ("encode_sub_floor", "code = (int)nearbyint(a * 512.0);", "code = (int)floor(a * 512.0);"),
 ("encode_sub_thresh", "if (a < ldexp(1.0, -6))", "if (a < ldexp(1.0, -7))"),
 ("encode_nosign", "sign = signbit(x) ? 0x80 : 0x00;", "sign = 0x00;"),
 ("encode_nan", "return 0x7F;\n    sign", "return 0x7E;\n    sign"),
 ("bf16_round_floor", "ldexp(nearbyint(ldexp(m, 8)), e - 8)", "ldexp(floor(ldexp(m, 8)), e - 8)"),
 ("k_no_interleave", "2 * (int64_t)e + (t & 1);", "2 * (int64_t)e + 0 * (t & 1);"),
 ("k_transposed_pair", "return pair_row * (2 * (int64_t)D) + 2 * (int64_t)e + (t & 1);",
  "return pair_row * (2 * (int64_t)D) + (int64_t)e + (int64_t)D * (t & 1);"),
 ("v_transposed", "return ((pb * Hkv + h) * (int64_t)B + t) * (int64_t)D + e;",
  "return ((pb * Hkv + h) * (int64_t)D + e) * (int64_t)B + t;"),
 ("k_layout_flip", "if (sh->k_layout == 0)", "if (sh->k_layout != 0)"),
 ("rope32_sign1", "out[e] = ac - bs;", "out[e] = ac + bs;"),
 ("rope32_sign2", "out[e + half] = bc + as;", "out[e + half] = bc - as;"),
 ("rope32_interleaved", "float a = x[e], b = x[e + half];", "float a = x[2 * e], b = x[2 * e + 1];"),
 ("rope64_sign", "out[e] = a * c - b * s;", "out[e] = a * c + b * s;"),
 ("rope64_interleaved", "double a = x[e], b = x[e + half], c", "double a = x[2 * e], b = x[2 * e + 1], c"),
 ("rope64_cos_sin_swap", "c = (double)cs[e], s = (double)sn[e];", "c = (double)sn[e], s = (double)cs[e];"),
 ("append_kscale_mul", "float kq = kr[e] / k_scale[i];", "float kq = kr[e] * k_scale[i];"),
 ("append_vscale_k", "float vq = bf16_to_f32(vr16[e]) / v_scale[i];", "float vq = bf16_to_f32(vr16[e]) / k_scale[i];"),
 ("append_slot_swap", "slot = layer_is_swa(i) ? upd_swa[b] : upd_full[b];", "slot = layer_is_swa(i) ? upd_full[b] : upd_swa[b];"),
 ("append_group_mod", "int32_t j = i / 2;\n        for (int32_t b", "int32_t j = i % (NL / 2);\n        for (int32_t b"),
 ("append_no_active", "if (!active[b])\n                continue;\n            slot", "slot"),
 ("append_rope_row0", "ora_rope_f32(kin, cosb + (int64_t)b * half, sinb + (int64_t)b * half, D, kr);",
  "ora_rope_f32(kin, cosb, sinb, D, kr);"),
 ("append_no_rope", "for (int32_t e = 0; e < D; ++e) {\n                    float kq = kr[e]",
  "for (int32_t e = 0; e < D; ++e) {\n                    float kq = kin[e]"),
 ("append_krow_batch_major", "const uint16_t *kr16 = k_new + (((int64_t)i * Bt + b) * Hkv + h) * D;",
  "const uint16_t *kr16 = k_new + (((int64_t)b * NL + i) * Hkv + h) * D;"),
 ("append_t_swap", "t = (int32_t)(slot % B);", "t = (int32_t)(slot % B) ^ 1;"),
 ("parity_flip", "return (i % 2) == 0;", "return (i % 2) == 1;"),
 ("window_off_by_one", "*lo = pw - sh->window + 1;", "*lo = pw - sh->window;"),
 ("window_hi", "*hi = pw;", "*hi = pw - 1;"),
 ("full_hi", "*hi = in->pos[b];", "*hi = in->pos[b] - 1;"),
 ("swa_uses_pos", "int64_t pw = in->pos_w[b];", "int64_t pw = in->pos[b];"),
 ("gqa_interleaved", "int32_t h = kvh * G + g;", "int32_t h = g * sh->num_kv_heads + kvh;"),
 ("q_rope_row0", "ora_rope_f64(qd, in->cosb + (int64_t)b * (D / 2), in->sinb + (int64_t)b * (D / 2), D, qr + (int64_t)g * D);",
  "ora_rope_f64(qd, in->cosb, in->sinb, D, qr + (int64_t)g * D);"),
 ("q_no_rope", "ora_rope_f64(qd, in->cosb + (int64_t)b * (D / 2), in->sinb + (int64_t)b * (D / 2), D, qr + (int64_t)g * D);",
  "memcpy(qr + (int64_t)g * D, qd, sizeof(double) * D);"),
 ("load_k_vscale", "* (double)in->k_scale[i];", "* (double)in->v_scale[i];"),
 ("load_v_noscale", "* (double)in->v_scale[i];\n    }", ";\n    }"),
 ("load_token_swap", "int32_t off = (int32_t)(t % B);", "int32_t off = (int32_t)(t % B) ^ 1;"),
 ("inv_d", "1.0 / sqrt((double)D)", "1.0 / (double)D"),
 ("no_scale", "sc[(t - lo) * G + g] = s * inv_sqrt_d;", "sc[(t - lo) * G + g] = s;"),
 ("score_head0", "s += qr[(int64_t)g * D + e] * kk[e];", "s += qr[e] * kk[e];"),
 ("pv_uses_k", "+= w * vv[e];", "+= w * kk[e];"),
 ("chunk_drop", "c1 = lo + (n * (s + 1)) / nsplit;", "c1 = lo + (n * (s + 1)) / nsplit - (s + 1 < nsplit);"),
 ("merge_L_norescale", "L += exp(ms[s * G + g] - M) * ls[s * G + g];", "L += ls[s * G + g];"),
 ("merge_acc_norescale", "acc += exp(ms[s * G + g] - M) * os[((int64_t)s * G + g) * D + e];", "acc += os[((int64_t)s * G + g) * D + e];"),
 ("sink_index", "sinks[(int64_t)i * sh->num_q_heads + (int64_t)kvh * G + g]", "sinks[(int64_t)i * sh->num_q_heads + g]"),
 ("sink_layer", "sinks[(int64_t)i * sh->num_q_heads + (int64_t)kvh * G + g]", "sinks[(int64_t)kvh * G + g]"),
 ("sink_unshifted", "L += exp(sink - M);", "L += exp(sink);"),
 ("sink_dropped", "L += exp(sink - M);", "L += 0.0;"),
 ("inactive_attends", "if (!in->active[b])\n        return 0;\n    key_range", "key_range"),
 ("stack_out_batch_major", "double *o = out + ((((int64_t)i * Bt + b) * Hq) + (int64_t)kvh * G) * D;",
  "double *o = out + ((((int64_t)b * NL + i) * Hq) + (int64_t)kvh * G) * D;"),
 ("stack_v_group_rev", "in.vbuf = v_bufs[i / 2];", "in.vbuf = v_bufs[(NL / 2 - 1) - i / 2];"),
 ("stack_k_group_rev", "in.kbuf = k_bufs[i / 2];", "in.kbuf = k_bufs[(NL / 2 - 1) - i / 2];"),
 ("stack_out_head_offset", "+ (int64_t)kvh * G) * D;", "+ (int64_t)kvh) * D;"),
 ("regions_nodedup", "if (out[k] == two[h])\n                    seen = 1;", "if (out[k] == two[h])\n                    seen = 0;"),
 ("regions_v_first", "two[0] = bases_k[i];\n        two[1] = bases_v[i];", "two[0] = bases_v[i];\n        two[1] = bases_k[i];"),
 ("ingest_swap", "regions[r][(int64_t)b * block_len + x] = src[d * block_len + x];",
  "regions[r][(int64_t)b * block_len + x] = src[(int64_t)b * block_len + x];"),
 ("di_full_N", "*full_count = (N - 1 + B - 1) / B;", "*full_count = (N + B - 1) / B;"),
 ("di_first_plus1", "int64_t first_key = N - W > 0 ? N - W : 0;", "int64_t first_key = N - W + 1 > 0 ? N - W + 1 : 0;"),
 ("di_last_N1", "int64_t last_key = N - 2;", "int64_t last_key = N - 1;"),
]


def _tree(tmp_path, text: str) -> str:
    """A copy of the oracle (with `text` as its C source) and of the tests,
    beside links to the input generators, the package and its header."""
    d = str(tmp_path / "tree")
    skip = shutil.ignore_patterns("_build", "__pycache__")
    shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(d, "oracle"), ignore=skip)
    shutil.copytree(os.path.join(ROOT, "tests"), os.path.join(d, "tests"), ignore=skip)
    for name in ("gk_inputs", "paged_fp8_kv_gk_gb300", "include"):
        os.symlink(os.path.join(ROOT, name), os.path.join(d, name))
    with open(os.path.join(d, "oracle", "gk_oracle.c"), "w") as f:
        f.write(text)
    subprocess.check_call([sys.executable, "-c", "import oracle; oracle.build(force=True)"], cwd=d)
    return d


def _run_pins(d: str) -> subprocess.CompletedProcess:
    cmd = [sys.executable, "-m", "pytest", *PIN_TESTS, "-q", "-x", "-p", "no:cacheprovider",
           "-k", NOT_PINS]
    return subprocess.run(cmd, cwd=d, capture_output=True, text=True, timeout=3600)


def test_unmutated_copy_passes(tmp_path):
    r = _run_pins(_tree(tmp_path, SRC))
    assert r.returncode == 0, r.stdout[-3000:]


@pytest.mark.parametrize("label,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, label, old, new):
    assert SRC.count(old) == 1, label
    r = _run_pins(_tree(tmp_path, SRC.replace(old, new)))
    # 1: some pin failed; a negative code: the mutant crashed the test process
    assert r.returncode == 1 or r.returncode < 0, (label, r.returncode, r.stdout[-2000:])
