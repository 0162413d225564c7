"""Pins of the oracle's extend-path gather (c7) and gather-then-cast (c8) against values fixed by the
formats and by plain indexing: a lossless FP8 -> NVFP4 -> FP8 round trip, saturation, zero scales,
the global scale's single rounding, bad page ids, and the page-table walk."""
import numpy as np

import oracle

E4M3_MAX, E4M3_NEG_MAX = 0x7E, 0xFE


def _pool_from_tokens(tokens_fp8, page_size=64):
    """NVFP4 pool (g = 1) of whole pages holding the given FP8 token rows, page-major."""
    n = tokens_fp8.shape[0]
    data, scale = oracle.quant_tokens(tokens_fp8, oracle.SRC_FP8, oracle.KV_NVFP4, 1.0)
    pages = n // page_size
    return data.reshape(pages, page_size, 288), scale.reshape(pages, page_size, 36)


def test_lossless_round_trip_restores_the_fp8_bytes():
    # Blocks whose values are (E4M3 scale s) x (E2M1 values) with amax = 6 s quantize to NVFP4 exactly,
    # and the FP8 workspace must give back the original bytes.
    rng = np.random.default_rng(1)
    e2m1 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)
    scales = np.array([2.0 ** k for k in range(-6, 5)], np.float64)     # powers of two: exact in E4M3
    tokens = np.zeros((128, 576), np.float64)
    for t in range(128):
        for b in range(36):
            s = scales[rng.integers(len(scales))]
            v = e2m1[rng.integers(0, 8, 16)] * np.where(rng.integers(0, 2, 16) == 1, -1.0, 1.0)
            v[rng.integers(16)] = 6.0          # amax = 6 s makes the block scale exactly s
            tokens[t, 16 * b:16 * b + 16] = v * s
    fp8 = oracle.encode_array(tokens.astype(np.float32).ravel(), 1).reshape(128, 576)
    # every value is exactly representable in E4M3 (at most 3 significant bits, in range)
    assert np.array_equal(np.vectorize(oracle.e4m3_value)(fp8), tokens)
    data, scale = _pool_from_tokens(fp8)
    ws, bad = oracle.gather_fp8(data, scale, oracle.KV_NVFP4, 1.0, 64, 2, [0, 2], [1, 0], [0, 128])
    assert bad == 0
    assert np.array_equal(ws[:64], fp8[64:]) and np.array_equal(ws[64:], fp8[:64])


def test_saturation_zero_scale_and_signs():
    data = np.zeros((1, 64, 288), np.uint8)
    scale = np.zeros((1, 64, 36), np.uint8)
    scale[0, 0, 0] = 0x7E                     # block scale 448
    data[0, 0, 0] = 0x7 | (0xF << 4)          # codes +6 and -6: |448 * 6| = 2688 > 448
    data[0, 0, 1] = 0x2                       # code +1: 448
    scale[0, 0, 1] = 0x00                     # block scale 0: every code gives 0
    data[0, 0, 8] = 0x77
    ws, _ = oracle.gather_fp8(data, scale, oracle.KV_NVFP4, 1.0, 64, 1, [0, 1], [0], [0, 1])
    assert ws[0, 0] == E4M3_MAX and ws[0, 1] == E4M3_NEG_MAX and ws[0, 2] == E4M3_MAX
    assert np.all(ws[0, 16:32] == 0)


def test_global_scale_is_one_fp32_rounding():
    rng = np.random.default_rng(2)
    data = rng.integers(0, 256, (1, 64, 288), dtype=np.uint8)
    scale = rng.integers(0, 0x70, (1, 64, 36), dtype=np.uint8)
    for g in (1.0, 0.5, 2.0 ** -7, 0.1234):
        ws, _ = oracle.gather_fp8(data, scale, oracle.KV_NVFP4, g, 64, 1, [0, 1], [0], [0, 64])
        # independent statement: e4m3(float32(float32(s * e) * float32(g))) per element
        for t in (0, 17, 63):
            for i in range(0, 576, 7):
                byte = data[0, t, i // 2]
                code = (byte >> 4) if i & 1 else (byte & 0xF)
                se = np.float32(oracle.e4m3_value(int(scale[0, t, i // 16])) * oracle.e2m1_value(int(code)))
                v = np.float32(se * np.float32(g))
                assert ws[t, i] == oracle.e4m3_encode(float(v))
        if g == 0.5:     # halving moves every nonzero, unsaturated, normal value down one binade
            ws1, _ = oracle.gather_fp8(data, scale, oracle.KV_NVFP4, 1.0, 64, 1, [0, 1], [0], [0, 64])
            v1 = np.vectorize(oracle.e4m3_value)(ws1)
            vh = np.vectorize(oracle.e4m3_value)(ws)
            m = (np.abs(v1) >= 2.0 ** -5) & (np.abs(v1) < 448)
            assert np.array_equal(vh[m], v1[m] / 2)


def test_fp8_pool_gather_is_plain_indexing_and_bad_pages_are_zero():
    rng = np.random.default_rng(3)
    pool = rng.integers(0, 256, (6, 64, 576), dtype=np.uint8)
    lens = np.array([130, 0, 64, 5])
    indptr = np.array([0, 3, 3, 4, 5])
    indices = np.array([4, 1 << 20, 2, 0, 5], np.int32)      # second page of request 0 is outside the pool
    tok = np.concatenate([[0], np.cumsum(lens)])
    ws, bad = oracle.gather_fp8(pool, None, oracle.KV_FP8, 1.0, 64, 6, indptr, indices, tok)
    flat = pool.reshape(-1, 576)
    expect = []
    for r in range(4):
        for t in range(lens[r]):
            p = indices[indptr[r] + t // 64]
            expect.append(flat[p * 64 + t % 64] if p < 6 else np.zeros(576, np.uint8))
    assert np.array_equal(ws, np.array(expect))
    assert bad == 64                      # tokens 64..127 of request 0


def test_gather_pages_bf16_is_the_cast_of_the_selected_pages():
    rng = np.random.default_rng(4)
    pool = rng.integers(0, 256, (5, 64, 576), dtype=np.uint8)
    ids = np.array([3, 0, 9, 3], np.int32)
    out = oracle.gather_pages_bf16(pool, ids)
    assert np.array_equal(out[0], oracle.cast_fp8_to_bf16(pool[3]))
    assert np.array_equal(out[1], oracle.cast_fp8_to_bf16(pool[0]))
    assert np.all(out[2] == 0) and np.array_equal(out[3], out[0])
    # a BF16 value widened to float equals the FP8 value (exact cast), except NaN bytes
    f = (out[1].astype(np.uint32) << 16).view(np.float32)
    v = np.vectorize(oracle.e4m3_value)(pool[0])
    ok = (pool[0] & 0x7F) != 0x7F
    assert np.array_equal(f[ok].astype(np.float64), v[ok])
