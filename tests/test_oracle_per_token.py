"""Pins of the oracle's per-token-scaled FP8 layout (c9): each token's 576 E4M3 codes carry one FP32
scale of their own, 64 tokens per page, the codes of a page first and its scales after them. The
layout is the pages' indexer key cache ("The Precision Frontier: Implementing bf16 Index Keys ...",
section "The Message: Planning the bf16-K Implementation": 128 elements + 4 scale bytes = 132 bytes per
token, a paged [npages, page_bytes] uint8 buffer, page size 64) applied to the 576-wide latent.

Pinned by: the byte layout of a page; the largest magnitude mapping onto 448; exact invariance of the
codes under power-of-two rescaling of a token (the scale follows, the codes do not move); the reduction
to the plain E4M3 codec (c2) when the scale is 1; zero and NaN tokens; the E4M3 rounding bound; and
attention over such a pool against torch's float64 attention on values rebuilt from the bytes with
torch's own E4M3 table."""
import numpy as np
import pytest
import torch

import oracle
import synth

PT = oracle.KV_FP8_PT


def _bf16_tokens(rng, n, scale=1.0):
    x = (rng.standard_normal((n, 576)) * scale).astype(np.float32)
    x[:, rng.integers(0, 576, 4)] *= 20.0
    return (x.view(np.uint32) >> 16).astype(np.uint16)          # BF16 bits (truncation is fine here)


def _bf16_to_f32(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _e4m3_torch(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_page_layout():
    assert oracle.PAGE_BYTES_PT == 64 * 580 == 37120
    rng = np.random.default_rng(1)
    src = _bf16_tokens(rng, 3)
    pool = oracle.pt_pool(5)
    slots = np.array([3 * 64 + 5, 0, 4 * 64 + 63], np.int64)
    oracle.append(src, oracle.SRC_BF16, slots, PT, 1.0, 64, 5, pool, None)
    codes, sig = oracle.quant_tokens(src, oracle.SRC_BF16, PT)
    for t, s in enumerate(slots):
        page, off = divmod(int(s), 64)
        assert np.array_equal(pool[page, off * 576:(off + 1) * 576], codes[t])
        assert pool[page, 64 * 576 + 4 * off:64 * 576 + 4 * off + 4].view(np.float32)[0] == sig[t]
    touched = np.zeros_like(pool, bool)
    for s in slots:
        page, off = divmod(int(s), 64)
        touched[page, off * 576:(off + 1) * 576] = True
        touched[page, 64 * 576 + 4 * off:64 * 576 + 4 * off + 4] = True
    assert not pool[~touched].any()


def test_largest_magnitude_maps_to_448():
    rng = np.random.default_rng(2)
    src = _bf16_tokens(rng, 64)
    codes, sig = oracle.quant_tokens(src, oracle.SRC_BF16, PT)
    x = _bf16_to_f32(src)
    amax = np.abs(x).max(1)
    assert np.array_equal(sig, (amax / np.float32(448.0)).astype(np.float32))
    for t in range(64):
        i = int(np.abs(x[t]).argmax())
        assert codes[t, i] == (0x7E if x[t, i] > 0 else 0xFE)
        assert (codes[t] & 0x7F).max() == 0x7E


@pytest.mark.parametrize("k", [-20, -3, 1, 7, 30])
def test_power_of_two_rescaling_moves_only_the_scale(k):
    rng = np.random.default_rng(3)
    src = _bf16_tokens(rng, 32)
    x = _bf16_to_f32(src)
    y = (x * np.float32(2.0 ** k)).astype(np.float32)
    src2 = (y.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(_bf16_to_f32(src2), y)                # exact in BF16
    c1, s1 = oracle.quant_tokens(src, oracle.SRC_BF16, PT)
    c2, s2 = oracle.quant_tokens(src2, oracle.SRC_BF16, PT)
    assert np.array_equal(c1, c2)
    assert np.array_equal(s2, (s1 * np.float32(2.0 ** k)).astype(np.float32))


def test_unit_scale_is_the_plain_e4m3_codec():
    rng = np.random.default_rng(4)
    x = rng.uniform(-448, 448, (8, 576)).astype(np.float32)
    x[:, 7] = 448.0
    src = (x.view(np.uint32) >> 16).astype(np.uint16)
    xf = _bf16_to_f32(src)
    codes, sig = oracle.quant_tokens(src, oracle.SRC_BF16, PT)
    assert np.all(sig == 1.0)
    assert np.array_equal(codes, oracle.encode_array(xf, 1).reshape(8, 576))


def test_zero_and_nan_tokens():
    src = np.zeros((2, 576), np.uint16)
    src[0, 10] = 0x8000                                          # -0
    src[1, 3] = 0x7FC0                                           # NaN
    src[1, 4] = 0x3F80                                           # 1.0
    codes, sig = oracle.quant_tokens(src, oracle.SRC_BF16, PT)
    assert sig[0] == 0.0 and codes[0, 10] == 0x80 and not np.delete(codes[0], 10).any()
    assert sig[1:2].view(np.uint32)[0] == 0x7FC00000 and np.all(codes[1] == 0x7F)


def test_rounding_bound():
    rng = np.random.default_rng(5)
    src = _bf16_tokens(rng, 128, scale=3.0)
    codes, sig = oracle.quant_tokens(src, oracle.SRC_BF16, PT)
    x = _bf16_to_f32(src).astype(np.float64)
    xh = sig[:, None].astype(np.float64) * _e4m3_torch(codes)
    u = np.abs(x) / sig[:, None]
    normal = u >= 2.0 ** -6
    assert np.all(np.abs(x - xh)[normal] <= 2.0 ** -4 * np.abs(x)[normal] * (1 + 1e-6))
    assert np.all(np.abs(x - xh)[~normal] <= (sig[:, None] * 2.0 ** -10 * (1 + 1e-6) * np.ones_like(x))[~normal])
    for t in range(3):                                           # the oracle's dequant reads the page
        pool = oracle.pt_pool(2)
        oracle.append(src[t:t + 1], oracle.SRC_BF16, np.array([64 + 9 * t], np.int64), PT, 1.0, 64, 2, pool, None)
        assert np.array_equal(oracle.dequant_slot(pool, None, PT, 1.0, 64 + 9 * t), xh[t])


@pytest.mark.parametrize("lens", [[256], [1, 64, 65, 200]])
def test_attention_matches_torch_sdpa_float64(lens):
    w = synth.build_workload("pt", lens, heads=16, pool_pages=16, seed=6, outliers=2)
    pool = oracle.pt_pool(w.num_pages)
    src = w.src_fp8.numpy()
    oracle.append(src, oracle.SRC_FP8, w.slots.numpy(), PT, 1.0, 64, w.num_pages, pool, None)
    qb = w.q.view(torch.int16).numpy().view(np.uint16)
    o, lse = oracle.mla_decode(qb, pool, None, PT, 64, w.num_pages, w.kv_indptr, w.kv_indices, w.kv_len,
                               w.sm_scale, 1.0)
    sm = float(np.float32(w.sm_scale))
    for r, L in enumerate(lens):
        t = np.arange(L)
        pages = w.kv_indices[w.kv_indptr[r] + t // 64]
        rows = np.stack([pool[p, (i % 64) * 576:(i % 64 + 1) * 576] for p, i in zip(pages, t)])
        sig = np.array([pool[p, 64 * 576 + 4 * (i % 64):64 * 576 + 4 * (i % 64) + 4].view(np.float32)[0]
                        for p, i in zip(pages, t)], np.float64)
        x = torch.from_numpy(sig[:, None] * _e4m3_torch(rows))
        q = w.q[r].to(torch.float64)
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[None, :, None, :], x[None, None].expand(1, 16, L, 576), x[None, None, :, :512].expand(1, 16, L, 512),
            scale=sm)[0, :, 0, :]
        assert torch.allclose(torch.from_numpy(o[r * 16:(r + 1) * 16]), ref, rtol=1e-12, atol=1e-12)
        z = sm * (q @ x.T)
        assert np.allclose(lse[r * 16:(r + 1) * 16], torch.logsumexp(z, dim=1).numpy(), rtol=0, atol=1e-12)
