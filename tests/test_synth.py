"""The shared input generator: SplitMix64 against its scalar definition, determinism, and the
layout of the generated workloads (CSR page table, poisoned unowned slots, length recipe)."""
import numpy as np
import torch

import synth


def test_splitmix64_matches_scalar_definition():
    key = synth.stream_key(0, "latent")
    c = torch.arange(0, 1000, 37, dtype=torch.int64)
    got = synth.raw64(key, c).numpy().view(np.uint64)
    for i, ci in enumerate(c.tolist()):
        x = (key + (ci + 1) * 0x9E3779B97F4A7C15) & ((1 << 64) - 1)
        assert int(got[i]) == synth.splitmix64_int(x)
    # the published first output of SplitMix64 seeded with 0 (state += golden, then mix)
    assert synth.splitmix64_int(0x9E3779B97F4A7C15) == 0xE220A8397B1DCDAF


def test_uniform_and_normal_moments():
    key = synth.stream_key(1, "misc")
    u = synth.uniform(key, torch.arange(200000, dtype=torch.int64))
    assert 0 < float(u.min()) and float(u.max()) < 1
    assert abs(float(u.mean()) - 0.5) < 0.005
    n = synth.normal_pairs(key, torch.arange(100000, dtype=torch.int64)).reshape(-1)
    assert abs(float(n.mean())) < 0.01 and abs(float(n.std()) - 1) < 0.01


def test_workload_is_deterministic_and_page_table_is_consistent():
    a = synth.build_workload("t", [256, 5, 64], heads=16, pool_pages=10, seed=3, outliers=4)
    b = synth.build_workload("t", [256, 5, 64], heads=16, pool_pages=10, seed=3, outliers=4)
    assert torch.equal(a.pool_fp8, b.pool_fp8) and torch.equal(a.q, b.q)
    assert a.kv_indptr.tolist() == [0, 4, 5, 6]
    assert len(set(a.kv_indices.tolist())) == 6 and max(a.kv_indices) < 10
    flat = a.pool_fp8.view(-1, 576)
    owned = set(a.slots.tolist())
    assert len(owned) == 325
    for s in range(640):
        if s not in owned:
            assert bool((flat[s] == synth.FP8_NAN).all())
    assert torch.equal(flat[a.slots], a.src_fp8)
    assert len(a.outliers) == 4 and len(set(a.outliers)) == 4


def test_tiny_workload_recipe():
    w = synth.workload("mla_tiny_b1_h16_l256")
    assert w.batch == 1 and w.heads == 16 and w.num_pages == 8 and w.kv_len.tolist() == [256]
    assert w.kv_indices.tolist() == synth.seeded_perm(0, "perm", 8)[:4].tolist()
    assert abs(w.sm_scale - 192 ** -0.5) < 1e-15
    x = w.src_fp8.view(torch.float8_e4m3fn).to(torch.float32)
    assert abs(float(x.std()) - 1) < 0.05


def test_mixed_lengths_recipe():
    lens, raw = synth.log_uniform_lengths(0, 64, 512, 65536, 495552)
    assert raw.min() >= 512 and raw.max() <= 65536
    assert lens.sum() <= 0.9 * 495552 + 64 and lens.min() >= 1
    assert np.sum((lens + 63) // 64) <= 495552 // 64
