"""Pins for the oracle's E4M3 codec, packed layout and RoPE (CPU only).

Each check ties the oracle to something other than itself: the OCP E4M3 table,
torch's float8_e4m3fn conversion (a library routine), a brute-force nearest
search over the code table, torch's own .view() indexing of the page's packed
shape, complex multiplication for the rotation, and the byte counts printed in
"GPT-OSS-120B giga-kernel decode", section "KV budget".
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ------------------------------------------------------------------ P1 decode
def test_decode_matches_ocp_table():
    for code_hex, val in _golden_rows("e4m3_values.txt"):
        got = oracle.e4m3_decode(np.array([int(code_hex, 16)], np.uint8))[0]
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))


def test_decode_all_codes_vs_torch_float8():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(ours), nan)
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(ours[~nan], lib[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(lib[~nan]))


# ------------------------------------------------------------------ P2 encode
_POS_VALS = np.array([float(v) for v in oracle.e4m3_decode(np.arange(127, dtype=np.uint8))])


def _brute_encode(x):
    """Nearest finite E4M3 code by search over the sorted value table, ties to
    the even code, |x| > 448 -> 448, NaN -> 0x7F."""
    x = np.asarray(x, np.float32)
    a = np.abs(x.astype(np.float64))
    idx = np.searchsorted(_POS_VALS, a)          # first value >= a
    hi = np.minimum(idx, 126)
    lo = np.maximum(idx - 1, 0)
    dlo = np.abs(a - _POS_VALS[lo])
    dhi = np.abs(_POS_VALS[hi] - a)
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    pick = np.where(a > 448.0, 126, pick).astype(np.uint8)
    code = pick | np.where(np.signbit(x), 0x80, 0).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)


def test_encode_exhaustive_relevant_range():
    """Every fp32 bit pattern with |x| in [2^-12, 2^10), both signs (about
    3.5e8 values, checked exponent by exponent)."""
    mant = np.arange(1 << 23, dtype=np.uint32)
    for e in range(127 - 12, 127 + 10):
        for s in (0, 1):
            bits = (np.uint32(s) << np.uint32(31)) | (np.uint32(e) << np.uint32(23)) | mant
            x = bits.view(np.float32)
            got = oracle.e4m3_encode(x)
            exp = _brute_encode(x)
            bad = np.nonzero(got != exp)[0]
            assert bad.size == 0, (e, s, x[bad[:5]], got[bad[:5]], exp[bad[:5]])


def test_encode_outside_that_range_is_zero_or_saturated():
    """The rest of the fp32 bit patterns, by closed form (OCP E4M3 fn, RNE,
    satfinite): |x| < 2^-12 lies below half the smallest subnormal (2^-10)
    and encodes to a zero of the same sign; |x| >= 2^10 (infinities included)
    lies past 448 and encodes to +-448 (0x7E / 0xFE); NaNs encode to 0x7F.
    Every exponent field is visited with a strided sample of its mantissas
    plus both ends."""
    mant = np.unique(np.concatenate([np.arange(0, 1 << 23, 4099, dtype=np.uint32),
                                     np.array([0, 1, (1 << 23) - 1], np.uint32)]))
    for e in list(range(0, 127 - 12)) + list(range(127 + 10, 256)):
        for s in (0, 1):
            bits = (np.uint32(s) << np.uint32(31)) | (np.uint32(e) << np.uint32(23)) | mant
            x = bits.view(np.float32)
            got = oracle.e4m3_encode(x)
            if e == 255:
                want = np.where(mant == 0, np.uint8(0x7E | (s << 7)), np.uint8(0x7F))
            elif e >= 127 + 10:
                want = np.full(mant.size, 0x7E | (s << 7), np.uint8)
            else:
                want = np.full(mant.size, s << 7, np.uint8)
            assert np.array_equal(got, want), (e, s)


def test_encode_random_bit_patterns_and_specials():
    rng = np.random.default_rng(123)
    bits = rng.integers(0, 1 << 32, size=1 << 22, dtype=np.uint64).astype(np.uint32)
    specials = np.array([0, 0x80000000, 0x7F800000, 0xFF800000, 0x7FC00000, 0xFFC00000, 1,
                         0x80000001, 0x00800000], np.uint32)
    x = np.concatenate([bits, specials]).view(np.float32)
    assert np.array_equal(oracle.e4m3_encode(x), _brute_encode(x))
    for v, c in ((np.inf, 0x7E), (-np.inf, 0xFE), (1e30, 0x7E), (448.0, 0x7E), (463.9, 0x7E),
                 (464.0, 0x7E), (2.0 ** -10, 0x00), (-(2.0 ** -10), 0x80)):
        assert oracle.e4m3_encode(np.array([v], np.float32))[0] == c


def test_encode_vs_torch_float8_in_range():
    """torch's float8_e4m3fn cast rounds to nearest even; inside +-448 it must
    agree with the oracle bit for bit."""
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.normal(0, s, 1 << 20) for s in (0.01, 1, 30, 150)]).astype(np.float32)
    x = np.clip(x, -448, 448).astype(np.float32)
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x), lib)


def test_encode_decode_roundtrip_all_finite_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


# ------------------------------------------------------------------ P3 layout
def test_packed_layout_golden_example():
    for row in _golden_rows("packed_k_example.txt"):
        pb, h, t, e, ko, vo = (int(v) for v in row)
        assert oracle.k_offset(2, 4, 3, pb, h, t, e) == ko
        assert oracle.v_offset(2, 4, 3, pb, h, t, e) == vo


@pytest.mark.parametrize("nb,Hkv,B,D", [(3, 2, 4, 3), (2, 8, 32, 64), (5, 1, 16, 64)])
def test_packed_layout_is_the_pages_view(nb, Hkv, B, D):
    """The offset formula equals indexing the page's trailing view
    [nb, kv, block//2, d, 2] of the [nb, kv, block, d] bytes (torch.view), and
    the map over all (pb, h, t, e) is a bijection onto the K half."""
    flat = torch.arange(nb * Hkv * B * D, dtype=torch.int64)
    view = flat.view(nb, Hkv, B // 2, D, 2)
    seen = np.zeros(flat.numel(), np.int64)
    for pb in range(nb):
        for h in range(Hkv):
            for t in range(B):
                for e in range(D):
                    off = oracle.k_offset(Hkv, B, D, pb, h, t, e)
                    assert off == int(view[pb, h, t // 2, e, t & 1])
                    seen[off] += 1
                    assert oracle.v_offset(Hkv, B, D, pb, h, t, e) == int(
                        flat.view(nb, Hkv, B, D)[pb, h, t, e])
    assert (seen == 1).all()


def test_kv_budget_numbers_printed_on_page():
    g = {r[0]: float(r[1]) for r in _golden_rows("kv_budget_gk.txt")}
    nb, kv, blk, d, groups = (int(g[k]) for k in ("num_blocks", "kv_heads", "block", "head_size",
                                                  "group_size"))
    per_buffer = 2 * nb * kv * blk * d  # [2, nb, kv, block, d] bytes, 1 B per FP8 element
    assert round(per_buffer * groups / 2 ** 30, 2) == g["kv_gib"]
    # the largest packed-K byte offset inside one group buffer stays under 2^32
    last = oracle.k_offset(kv, blk, d, nb - 1, kv - 1, blk - 1, d - 1)
    assert last == nb * kv * blk * d - 1 < 2 ** 32


# ------------------------------------------------------------------ P4 RoPE
def test_rope_identity_and_inverse():
    rng = np.random.default_rng(1)
    x = rng.normal(size=64)
    ones, zeros = np.ones(32, np.float32), np.zeros(32, np.float32)
    assert np.array_equal(oracle.rope_f64(x, ones, zeros), x)
    x32 = x.astype(np.float32)
    assert np.array_equal(oracle.rope_f32(x32, ones, zeros), x32)
    ang = rng.uniform(-10, 10, 32)
    c, s = np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)
    y = oracle.rope_f64(x, c, s)
    back = oracle.rope_f64(y, c, -s)
    # (c, s) are fp32-rounded, so c^2 + s^2 = 1 only to ~1e-7
    r2 = c.astype(np.float64) ** 2 + s.astype(np.float64) ** 2
    assert np.allclose(back, x * np.concatenate([r2, r2]), atol=1e-12)
    n0 = x[:32] ** 2 + x[32:] ** 2
    n1 = y[:32] ** 2 + y[32:] ** 2
    assert np.allclose(n1, n0 * r2, rtol=1e-12)


def test_rope_is_complex_rotation_of_half_pairs():
    rng = np.random.default_rng(2)
    x = rng.normal(size=64)
    ang = rng.uniform(-100, 100, 32)
    c, s = np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)
    z = (x[:32] + 1j * x[32:]) * (c.astype(np.float64) + 1j * s.astype(np.float64))
    y = oracle.rope_f64(x, c, s)
    assert np.allclose(y[:32], z.real, atol=1e-13) and np.allclose(y[32:], z.imag, atol=1e-13)
    # the fp32 path stays within fp32 rounding of the exact rotation
    y32 = oracle.rope_f32(x.astype(np.float32), c, s).astype(np.float64)
    z32 = (x.astype(np.float32)[:32].astype(np.float64) + 1j * x.astype(np.float32)[32:]) * (
        c.astype(np.float64) + 1j * s.astype(np.float64))
    assert np.allclose(y32[:32], z32.real, atol=1e-5) and np.allclose(y32[32:], z32.imag, atol=1e-5)


def test_round_bf16_vs_torch():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.normal(0, s, 100000) for s in (1e-3, 1, 1e3)])
    # torch rounds fp32 -> bf16 RNE; pick inputs exactly representable in fp32
    x = x.astype(np.float32).astype(np.float64)
    lib = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.round_bf16(x), lib)
