"""Pins of the oracle's dequant (c4), attention (c5) and LSE merge (c6): torch's float64
scaled-dot-product attention on tiny inputs, closed forms (L = 1, uniform weights, a dominant
logit), invariants (page permutation, weights summing to one), split-and-merge, and the
published E2M1 / torch E4M3 tables for the dequant."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.conftest import read_golden

FP8, NVFP4, BF16 = oracle.KV_FP8, oracle.KV_NVFP4, oracle.KV_BF16


def _qbits(q):
    return q.view(torch.int16).numpy().view(np.uint16)


def _fp8_values(pool_bytes):
    return torch.from_numpy(np.ascontiguousarray(pool_bytes)).view(torch.float8_e4m3fn).to(torch.float64)


def _gather_latent(w, r):
    """The request's latent rows in token order, straight from the FP8 pool bytes."""
    L = int(w.kv_len[r])
    t = np.arange(L)
    pages = w.kv_indices[w.kv_indptr[r] + t // 64]
    slots = pages.astype(np.int64) * 64 + t % 64
    return w.pool_fp8.view(-1, 576).numpy()[slots]


def _decode(w, kv_data, kv_scale, kv, g=1.0, sm_scale=None, pairs=None, lens=None):
    return oracle.mla_decode(_qbits(w.q), kv_data, kv_scale, kv, 64, w.num_pages, w.kv_indptr,
                             w.kv_indices, w.kv_len if lens is None else lens,
                             w.sm_scale if sm_scale is None else sm_scale, g, pairs)


@pytest.mark.parametrize("lens", [[256], [1, 64, 65, 200]])
def test_fp8_matches_torch_sdpa_float64(lens):
    w = synth.build_workload("t", lens, heads=16, pool_pages=16, seed=5, outliers=2)
    o, lse = _decode(w, w.pool_fp8.numpy(), None, FP8)
    sm = float(np.float32(w.sm_scale))
    for r, L in enumerate(lens):
        x = _fp8_values(_gather_latent(w, r))                       # [L, 576]
        q = w.q[r].to(torch.float64)                                # [H, 576]
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[None, :, None, :].expand(1, 16, 1, 576).reshape(1, 16, 1, 576),
            x[None, None].expand(1, 16, L, 576), x[None, None, :, :512].expand(1, 16, L, 512),
            scale=sm)[0, :, 0, :]
        got = torch.from_numpy(o[r * 16:(r + 1) * 16])
        assert torch.allclose(got, ref, rtol=1e-12, atol=1e-12)
        z = sm * (q @ x.T)
        assert np.allclose(lse[r * 16:(r + 1) * 16], torch.logsumexp(z, dim=1).numpy(), rtol=0, atol=1e-12)


def test_nvfp4_dequant_matches_tables():
    e2m1 = {int(c, 16): float(v) for c, v in read_golden("e2m1_codes.txt")}
    e4m3 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    rng = np.random.default_rng(7)
    data = rng.integers(0, 256, (3, 288), dtype=np.uint8)
    scales = rng.integers(0, 0x7F, (3, 36), dtype=np.uint8)
    for g in [1.0, 0.04464285820722580]:
        for slot in range(3):
            x = oracle.dequant_slot(data, scales, NVFP4, g, slot)
            for i in range(576):
                byte = data[slot, i // 2]
                code = (byte >> 4) if i % 2 else (byte & 0xF)
                want = g * e4m3[scales[slot, i // 16]] * e2m1[int(code)]
                assert x[i] == want


def test_nvfp4_decode_matches_sdpa_on_dequantised_latent():
    w = synth.build_workload("t", [130, 7], heads=16, pool_pages=8, seed=9, outliers=1)
    src = w.src_fp8.numpy()
    data = np.full((8 * 64, 288), 0xFF, np.uint8)
    scales = np.full((8 * 64, 36), 0x7F, np.uint8)
    g = float(np.float32(0.3))          # the oracle takes the global scale as FP32
    oracle.append(src, oracle.SRC_FP8, w.slots.numpy(), NVFP4, g, 64, 8, data, scales)
    o, lse = _decode(w, data, scales, NVFP4, g=g)
    row = 0
    for r, L in enumerate(w.kv_len):
        x = torch.tensor(np.stack([oracle.dequant_slot(data, scales, NVFP4, g, int(s))
                                   for s in w.slots.numpy()[row:row + L]]))
        row += L
        q = w.q[r].to(torch.float64)
        ref = torch.softmax(float(np.float32(w.sm_scale)) * (q @ x.T), dim=1) @ x[:, :512]
        assert np.allclose(o[r * 16:(r + 1) * 16], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_single_token_returns_its_value_rows():
    w = synth.build_workload("t", [1], heads=16, pool_pages=2, seed=1)
    o, lse = _decode(w, w.pool_fp8.numpy(), None, FP8)
    x = _fp8_values(_gather_latent(w, 0))[0]
    assert np.array_equal(o, np.tile(x[:512].numpy(), (16, 1)))
    z = float(np.float32(w.sm_scale)) * (w.q[0].to(torch.float64) @ x)
    assert np.allclose(lse, z.numpy(), atol=1e-13)


def test_zero_scale_gives_mean_and_log_length():
    w = synth.build_workload("t", [200], heads=16, pool_pages=4, seed=2)
    o, lse = _decode(w, w.pool_fp8.numpy(), None, FP8, sm_scale=0.0)
    x = _fp8_values(_gather_latent(w, 0))
    assert np.allclose(o, np.tile(x[:, :512].mean(0).numpy(), (16, 1)), rtol=1e-13, atol=1e-13)
    assert np.allclose(lse, math.log(200), atol=1e-13)


def test_weights_sum_to_one():
    # value dims all 1.0, rope dims random: logits differ, the output must be exactly 1 +- 1e-15
    w = synth.build_workload("t", [300], heads=16, pool_pages=5, seed=3)
    flat = w.pool_fp8.view(-1, 576)
    flat[:, :512] = 0x38                      # E4M3 1.0
    o, _ = _decode(w, w.pool_fp8.numpy(), None, FP8)
    assert np.max(np.abs(o - 1.0)) <= 1e-15 * 4


def test_dominant_logit_selects_its_token():
    w = synth.build_workload("t", [150], heads=16, pool_pages=3, seed=4)
    flat = w.pool_fp8.view(-1, 576)
    for s in w.slots.tolist():
        flat[s, 0] = 0x00
    hot = int(w.slots[77])
    flat[hot, 0] = 0x7E                      # 448
    w.q[:] = 0
    w.q[:, :, 0] = 1.0
    o, lse = _decode(w, w.pool_fp8.numpy(), None, FP8, sm_scale=0.25)   # logit gap 112
    want = _fp8_values(flat[hot].numpy()[None])[0, :512].numpy()
    assert np.allclose(o, np.tile(want, (16, 1)), rtol=0, atol=1e-30 + 1e-40)
    assert np.allclose(lse, 112.0, atol=1e-12)


def test_page_permutation_does_not_change_result():
    w = synth.build_workload("t", [64 * 5 + 9], heads=16, pool_pages=12, seed=6)
    o1, l1 = _decode(w, w.pool_fp8.numpy(), None, FP8)
    # move every page of the request somewhere else in the pool and rewrite the page table
    pool = w.pool_fp8.numpy().copy()
    new_pool = np.full_like(pool, 0x7F)
    free = [p for p in range(12) if p not in set(w.kv_indices.tolist())][::-1] + w.kv_indices.tolist()
    new_idx = np.array(free[:len(w.kv_indices)], np.int32)
    for old, new in zip(w.kv_indices, new_idx):
        new_pool[new] = pool[old]
    o2, l2 = oracle.mla_decode(_qbits(w.q), new_pool, None, FP8, 64, 12, w.kv_indptr, new_idx,
                               w.kv_len, w.sm_scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_split_and_lse_merge_equals_whole():
    w = synth.build_workload("t", [64 * 9 + 17], heads=16, pool_pages=12, seed=8, outliers=3)
    o, lse = _decode(w, w.pool_fp8.numpy(), None, FP8)
    L = int(w.kv_len[0])
    for cuts in ([0, 64, L], [0, 128, 320, 512, L], [0, 576, L]):
        parts_o, parts_l = [], []
        for a, b in zip(cuts[:-1], cuts[1:]):
            idx = w.kv_indices[a // 64: (b + 63) // 64]
            po, pl = oracle.mla_decode(_qbits(w.q), w.pool_fp8.numpy(), None, FP8, 64, 12,
                                       np.array([0, len(idx)], np.int32), idx,
                                       np.array([b - a], np.int32), w.sm_scale)
            parts_o.append(po)
            parts_l.append(pl)
        for h in range(16):
            mo, ml = oracle.lse_merge(np.stack([p[h] for p in parts_o]), np.array([p[h] for p in parts_l]))
            assert np.allclose(mo, o[h], rtol=1e-12, atol=1e-12) and abs(ml - lse[h]) < 1e-12


def test_merge_handles_empty_parts():
    o, l = oracle.lse_merge(np.zeros((2, 4)), np.array([-np.inf, -np.inf]))
    assert np.all(o == 0) and l == -np.inf
    o, l = oracle.lse_merge(np.array([[1.0, 2.0], [9.0, 9.0]]), np.array([0.5, -np.inf]))
    assert np.array_equal(o, [1.0, 2.0]) and l == 0.5


def test_empty_request_and_partial_page_masking():
    w = synth.build_workload("t", [0, 70], heads=16, pool_pages=4, seed=10, extra_pages=[1, 0])
    o, lse = _decode(w, w.pool_fp8.numpy(), None, FP8)
    assert np.all(o[:16] == 0) and np.all(lse[:16] == -np.inf)
    assert np.all(np.isfinite(o[16:])) and np.all(np.isfinite(lse[16:]))   # NaN poison after L unread


def test_bad_page_id_is_an_error():
    w = synth.build_workload("t", [10], heads=16, pool_pages=2, seed=11)
    bad = w.kv_indices.copy()
    bad[0] = 2
    with pytest.raises(ValueError):
        oracle.mla_decode(_qbits(w.q), w.pool_fp8.numpy(), None, FP8, 64, 2, w.kv_indptr, bad,
                          w.kv_len, w.sm_scale)


def test_bf16_pool_equals_fp8_pool():
    w = synth.build_workload("t", [100, 33], heads=16, pool_pages=6, seed=12, outliers=2)
    o8, l8 = _decode(w, w.pool_fp8.numpy(), None, FP8)
    bf = oracle.cast_fp8_to_bf16(w.pool_fp8.numpy())
    ob, lb = _decode(w, bf, None, BF16)
    assert np.array_equal(o8, ob) and np.array_equal(l8, lb)


def test_pairs_subset_matches_full():
    w = synth.build_workload("t", [90, 150], heads=16, pool_pages=6, seed=13)
    o, lse = _decode(w, w.pool_fp8.numpy(), None, FP8)
    pairs = np.array([[1, 3], [0, 15], [1, 0]], np.int32)
    os_, ls = _decode(w, w.pool_fp8.numpy(), None, FP8, pairs=pairs)
    for i, (r, h) in enumerate(pairs):
        assert np.array_equal(os_[i], o[r * 16 + h]) and ls[i] == lse[r * 16 + h]
