"""Pins of the oracle's number formats (c1-c3) against things other than the oracle itself:
the published E2M1 table, torch's float8_e4m3fn routines, brute-force nearest search, the page's
storage arithmetic, and invariants of the two-level scaling."""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.conftest import read_golden

E4M3_FINITE_POS = [c for c in range(0x7F)]          # 0x00..0x7E
E2M1_POS = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]  # re-derived below from the golden table


def test_e2m1_table_matches_published_table():
    rows = read_golden("e2m1_codes.txt")
    assert len(rows) == 16
    for code_s, val_s in rows:
        code, want = int(code_s, 16), float(val_s)
        got = oracle.e2m1_value(code)
        assert got == want and math.copysign(1, got) == math.copysign(1, want), (code, got, want)
    # what the pages fix: max magnitude 6 (block scale = amax / 6), 8 magnitudes, sign bit 0x8
    mags = sorted({abs(oracle.e2m1_value(c)) for c in range(16)})
    assert mags == E2M1_POS and max(mags) == 6.0


def test_e4m3_table_matches_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = oracle.e4m3_value(c)
        if np.isnan(ref[c]):
            assert np.isnan(got), c
        else:
            assert got == ref[c] and math.copysign(1, got) == math.copysign(1, ref[c]), (c, got, ref[c])
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e4m3_value(0x01) == 2.0 ** -9
    assert [c for c in range(256) if np.isnan(oracle.e4m3_value(c))] == [0x7F, 0xFF]


def _e4m3_sweep():
    vals = np.array([oracle.e4m3_value(c) for c in E4M3_FINITE_POS], dtype=np.float64)
    pts = [vals.astype(np.float32)]
    for a, b in zip(vals[:-1], vals[1:]):
        mid = np.float32((a + b) / 2)  # exact: e4m3 midpoints have few bits
        pts.append(np.array([mid, np.nextafter(mid, np.float32(0)), np.nextafter(mid, np.float32(1e9))],
                            dtype=np.float32))
        pts.append(np.linspace(a, b, 11, dtype=np.float64).astype(np.float32))
    rng = np.random.default_rng(0)
    pts.append(np.exp(rng.uniform(np.log(2.0 ** -14), np.log(448.0), 400000)).astype(np.float32))
    x = np.concatenate(pts)
    x = np.concatenate([x, -x])
    return x[np.abs(x) <= 448.0]


def test_e4m3_encode_matches_torch_rne_in_range():
    x = _e4m3_sweep()
    got = oracle.encode_array(x, 1)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(x[i]), int(got[i]), int(ref[i])) for i in bad[:10]]


def _nearest_even(x, values):
    """Brute force: index of the nearest value; on an exact tie, the even index."""
    d = np.abs(values[None, :] - x[:, None])
    best = d.min(axis=1)
    out = np.empty(x.size, dtype=np.int64)
    for i in range(x.size):
        cand = np.nonzero(d[i] == best[i])[0]
        ev = [c for c in cand if c % 2 == 0]
        out[i] = ev[0] if ev else cand[0]
    return out


def test_e4m3_encode_brute_force_midpoints():
    vals = np.array([oracle.e4m3_value(c) for c in E4M3_FINITE_POS], dtype=np.float64)
    x = np.abs(_e4m3_sweep()[:20000]).astype(np.float64)
    idx = _nearest_even(x, vals)
    got = oracle.encode_array(x.astype(np.float32), 1)
    assert np.array_equal(got, idx.astype(np.uint8))


def test_e4m3_saturation_nan_and_signed_zero():
    f = oracle.e4m3_encode
    for v in [448.0, 449.0, 464.0, 480.0, 1e6, float("inf"), 3.0e38]:
        assert f(v) == 0x7E and f(-v) == 0xFE
    assert f(float("nan")) == 0x7F and f(-float("nan")) == 0x7F
    assert f(0.0) == 0x00 and f(-0.0) == 0x80
    assert f(2.0 ** -11) == 0x00 and f(-(2.0 ** -11)) == 0x80      # below half the min subnormal
    assert f(2.0 ** -10) == 0x00                                   # tie 0 | 2^-9 -> even (0)
    assert f(3 * 2.0 ** -10) == 0x02                               # tie 1 | 2 (x 2^-9) -> even
    assert f(7.5 * 2.0 ** -9) == 0x08                              # tie into the first normal


def test_e4m3_round_trips():
    for c in list(range(0x7F)) + list(range(0x80, 0xFF)):
        v = oracle.e4m3_value(c)
        assert oracle.e4m3_encode(v) == c, hex(c)
        # E4M3 -> BF16 -> E4M3: the widening to BF16 is exact
        b = torch.tensor([v], dtype=torch.float32).to(torch.bfloat16).to(torch.float32).item()
        assert b == v and oracle.e4m3_encode(b) == c


def test_e2m1_encode_brute_force():
    vals = np.array(E2M1_POS)
    mids = (vals[:-1] + vals[1:]) / 2
    pts = [vals, mids, np.linspace(0, 8, 20001)]
    for m in mids:
        m32 = np.float32(m)
        pts.append(np.array([np.nextafter(m32, np.float32(0)), np.nextafter(m32, np.float32(9))], dtype=np.float64))
    x = np.concatenate(pts).astype(np.float32).astype(np.float64)
    idx = _nearest_even(np.minimum(x, 6.0), vals)   # saturate at 6
    got = oracle.encode_array(x.astype(np.float32), 2)
    assert np.array_equal(got, idx.astype(np.uint8))
    gotn = oracle.encode_array(-x.astype(np.float32), 2)
    assert np.array_equal(gotn, (idx | 8).astype(np.uint8))


def test_e2m1_ties_and_specials():
    f = oracle.e2m1_encode
    want = {0.25: 0x0, 0.75: 0x2, 1.25: 0x2, 1.75: 0x4, 2.5: 0x4, 3.5: 0x6, 5.0: 0x6, 6.0: 0x7,
            7.0: 0x7, 1e30: 0x7, float("inf"): 0x7}
    for v, c in want.items():
        assert f(v) == c and f(-v) == (c | 8), v
    assert f(float("nan")) == 0x0
    assert f(-0.1) == 0x8 and f(0.1) == 0x0


def test_storage_accounting_matches_page():
    g = {k: v for k, v in read_golden("nvfp4_storage.txt")}
    packed, scale = oracle.nvfp4_block(np.arange(16, dtype=np.float32), 1.0)
    assert packed.size == int(g["packed_bytes_per_block"]) and int(g["scale_bytes_per_block"]) == 1
    data, scales = oracle.quant_tokens(np.zeros((1, 576), np.uint8), oracle.SRC_FP8, oracle.KV_NVFP4)
    per_token = data.shape[1] + scales.shape[1]
    assert per_token == 324 == 576 * 9 // 16
    assert per_token / 576 == float(g["fraction_of_fp8"])
    assert round(576 / per_token, 2) == float(g["capacity_ratio_rounded"])


def _fp32(x):
    return np.float32(x)


def _block_check(x, g):
    """Brute-force check of one quantised block against the stated steps."""
    packed, s8 = oracle.nvfp4_block(x, g)
    x = x.astype(np.float32)
    amax = np.float32(np.max(np.abs(x)))
    s = _fp32(amax / _fp32(_fp32(6.0) * _fp32(g)))
    vals = np.array([oracle.e4m3_value(c) for c in E4M3_FINITE_POS])
    if s >= 448:
        want_s8 = 0x7E
    else:
        want_s8 = int(_nearest_even(np.array([float(s)]), vals)[0])
    assert s8 == want_s8, (float(s), s8, want_s8)
    sd = _fp32(_fp32(oracle.e4m3_value(s8)) * _fp32(g))
    codes = np.concatenate([(packed & 0xF)[:, None], (packed >> 4)[:, None]], axis=1).reshape(16)
    if sd == 0:
        assert np.all(codes == 0)
        return packed, s8
    q = (x / sd).astype(np.float32).astype(np.float64)
    mag = _nearest_even(np.minimum(np.abs(q), 6.0), np.array(E2M1_POS))
    want = np.where(np.signbit(q), mag | 8, mag)
    assert np.array_equal(codes, want.astype(np.uint8)), (x, codes, want)
    return packed, s8


def test_nvfp4_block_brute_force():
    rng = np.random.default_rng(1)
    for trial in range(400):
        g = [1.0, 0.25, 3.0, 120.0 / 2688.0][trial % 4]
        scale = np.exp(rng.uniform(-8, 6))
        x = (rng.standard_normal(16) * scale).astype(np.float32)
        if trial % 7 == 0:
            x[rng.integers(16)] *= 30
        _block_check(x, g)


def test_nvfp4_block_edge_cases():
    z = np.zeros(16, np.float32)
    packed, s8 = oracle.nvfp4_block(z, 1.0)
    assert s8 == 0 and not packed.any()
    neg0 = -z
    packed, s8 = oracle.nvfp4_block(neg0, 1.0)
    assert s8 == 0 and not packed.any()                 # zero-scale blocks give code 0x0
    tiny = np.full(16, 1e-6, np.float32)
    packed, s8 = oracle.nvfp4_block(tiny, 1.0)
    assert s8 == 0 and not packed.any()                 # scale rounds to zero
    nan = np.ones(16, np.float32)
    nan[3] = np.nan
    packed, s8 = oracle.nvfp4_block(nan, 1.0)
    assert s8 == 0x7F and not packed.any()              # NaN poisons the block scale
    big = np.full(16, 1e30, np.float32)
    big[0] = -1e30
    packed, s8 = oracle.nvfp4_block(big, 1.0)
    assert s8 == 0x7E and packed[0] == 0x7F             # scale saturates at 448, codes at +-6
    inf = np.ones(16, np.float32)
    inf[5] = np.inf
    packed, s8 = oracle.nvfp4_block(inf, 1.0)
    assert s8 == 0x7E and (packed[2] >> 4) == 0x7
    # amax = 6 * 2^k with g = 1: scale 2^k exactly, codes are exact E2M1 multiples
    x = np.array([6, -6, 4, 3, 2, 1.5, 1, 0.5, 0, -0.5, -1, -1.5, -2, -3, -4, 0], np.float32) * 0.125
    packed, s8 = oracle.nvfp4_block(x, 1.0)
    assert oracle.e4m3_value(s8) == 0.125
    dq = [oracle.e4m3_value(s8) * oracle.e2m1_value(c) for c in
          np.concatenate([(packed & 0xF)[:, None], (packed >> 4)[:, None]], 1).reshape(16)]
    assert np.array_equal(np.array(dq, np.float32), x)


def test_nvfp4_idempotent_when_scale_normal():
    rng = np.random.default_rng(2)
    n_checked = 0
    for _ in range(300):
        x = (rng.standard_normal(16) * np.exp(rng.uniform(-3, 4))).astype(np.float32)
        g = 1.0
        packed, s8 = oracle.nvfp4_block(x, g)
        sv = oracle.e4m3_value(s8)
        if not (2.0 ** -6 <= sv < 448):
            continue
        codes = np.concatenate([(packed & 0xF)[:, None], (packed >> 4)[:, None]], 1).reshape(16)
        dq = np.array([sv * g * oracle.e2m1_value(c) for c in codes], np.float32)
        p2, s2 = oracle.nvfp4_block(dq, g)
        if np.max(np.abs(dq)) == 0:
            continue
        # the re-derived scale may differ (amax of the dequantised block is 6*sv, 4*sv, ...);
        # requantisation must reproduce the same dequantised values
        c2 = np.concatenate([(p2 & 0xF)[:, None], (p2 >> 4)[:, None]], 1).reshape(16)
        dq2 = np.array([oracle.e4m3_value(s2) * g * oracle.e2m1_value(c) for c in c2], np.float32)
        assert np.array_equal(dq, dq2)
        n_checked += 1
    assert n_checked > 200


def test_quant_tokens_layout_and_bf16_source():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((5, 576)) * 3).astype(np.float32)
    bf = torch.from_numpy(x).to(torch.bfloat16)
    bits = bf.view(torch.int16).numpy().view(np.uint16)
    data, sc = oracle.quant_tokens(bits, oracle.SRC_BF16, oracle.KV_NVFP4, 1.0)
    xf = bf.to(torch.float32).numpy()
    for t in range(5):
        for j in range(36):
            p, s = oracle.nvfp4_block(xf[t, 16 * j:16 * j + 16], 1.0)
            assert np.array_equal(data[t, 8 * j:8 * j + 8], p) and sc[t, j] == s
    f8 = oracle.quant_tokens(bits, oracle.SRC_BF16, oracle.KV_FP8)
    ref = bf.to(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(f8, ref)   # |x| << 448: RNE agrees with torch


def test_append_writes_slots_and_skips_negative():
    rng = np.random.default_rng(4)
    src = torch.from_numpy(rng.standard_normal((4, 576)).astype(np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()
    pool = np.full((3 * 64, 288), 0xEE, np.uint8)
    scales = np.full((3 * 64, 36), 0xEE, np.uint8)
    slots = np.array([5, -1, 130, 64], np.int64)
    oracle.append(src, oracle.SRC_FP8, slots, oracle.KV_NVFP4, 1.0, 64, 3, pool, scales)
    d, s = oracle.quant_tokens(src, oracle.SRC_FP8, oracle.KV_NVFP4, 1.0)
    for i, sl in enumerate(slots):
        if sl >= 0:
            assert np.array_equal(pool[sl], d[i]) and np.array_equal(scales[sl], s[i])
    touched = {5, 130, 64}
    for sl in range(3 * 64):
        if sl not in touched:
            assert (pool[sl] == 0xEE).all()
    with pytest.raises(ValueError):
        oracle.append(src, oracle.SRC_FP8, np.array([0, 0, 0, 3 * 64], np.int64), oracle.KV_NVFP4,
                      1.0, 64, 3, pool, scales)


def test_cast_fp8_to_bf16_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.cast_fp8_to_bf16(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for c in range(256):
        if c in (0x7F, 0xFF):
            assert got[c] == 0x7FC0
        else:
            assert got[c] == ref[c], c
