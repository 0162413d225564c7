"""The token-major tcgen05 kernel (QKVP_ALGO_TCGEN05_TOKENS, 16-64 heads) against the FP64 oracle:
ragged batches split over different SM counts, every quantized pool dtype, forced rescales of the
running maxima, Q rows outside the FP16 range, and the full-size workloads at 16 / 32 / 64 heads in
the launch configuration the benchmark times."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import quantized_kv_paged_gb300 as q
import synth
from tests.helpers import compare, gpu_decode, gpu_pools, oracle_decode, oracle_pools

pytestmark = pytest.mark.gpu

FP8, NVFP4, FP8PT = q.KV_FP8_E4M3, q.KV_NVFP4, q.KV_FP8_PER_TOKEN
TM = q.ALGO_TCGEN05_TOKENS


def _run(w, kv, g=1.0, **kw):
    out, lse, plan = gpu_decode(w, kv, gpu_pools(w, kv, g), g, algo=TM, **kw)
    assert plan.algo == TM and plan.ctas_per_worker == 1
    o_ref, lse_ref = oracle_decode(w, kv, oracle_pools(w, kv, g), g, lens=kw.get("lens"))
    stats = compare(out.float().cpu().numpy().reshape(-1, 512), lse.cpu().numpy().reshape(-1), o_ref, lse_ref)
    return stats, plan


@pytest.mark.parametrize("heads", [16, 32, 48, 64])
@pytest.mark.parametrize("kv", [FP8, NVFP4, FP8PT])
def test_tm_ragged_batch_many_splits(qkvp, heads, kv):
    lens = [1, 63, 64, 65, 200, 0, 1000, 4097, 129]
    w = synth.build_workload("ragged_tm", lens, heads=heads, pool_pages=180, seed=90 + heads + kv, outliers=4,
                             device="cuda", extra_pages=[1] * len(lens))
    for sms in (4, 37, 152):
        _run(w, kv, g=0.37 if kv == NVFP4 else 1.0, num_sms=sms)


def test_tm_tiny_single_page(qkvp):
    w = synth.build_workload("one_tm", [17], heads=16, pool_pages=3, seed=3, device="cuda")
    _run(w, FP8, num_sms=2)


def test_tm_long_single_request_min_splits(qkvp):
    w = synth.build_workload("long_tm", [64 * 300 + 5], heads=64, pool_pages=320, seed=1, outliers=4,
                             device="cuda")
    stats, plan = _run(w, NVFP4, g=0.5, num_sms=16, min_splits=40)
    assert plan.num_segments >= 40


@pytest.mark.parametrize("heads", [16, 64])
def test_tm_lazy_rescale_of_running_max(qkvp, heads):
    """Late tokens whose logits jump far above the running maxima force O^T and the row sums to be
    rescaled, in some heads only."""
    w = synth.build_workload("rescale_tm", [64 * 12, 64 * 5 + 3], heads=heads, pool_pages=20, seed=9,
                             device="cuda")
    flat = w.pool_fp8.view(-1, 576)
    for r, tok in ((0, 64 * 9 + 7), (1, 64 * 4 + 1), (0, 64 * 11 + 63)):
        slot = int(w.kv_indices[w.kv_indptr[r] + tok // 64]) * 64 + tok % 64
        for ch in (3, 300, 560):
            flat[slot, ch] = 0x7E            # 448: the logit moves by tens
    _run(w, FP8, num_sms=2)                  # one segment per request: long runs of pages
    _run(w, FP8, num_sms=8)


@pytest.mark.parametrize("heads", [32, 64])
def test_tm_q_rows_outside_the_unscaled_fp16_range(qkvp, heads):
    lens = [300, 64, 1000]
    w = synth.build_workload("qrange_tm", lens, heads=heads, pool_pages=40, seed=11, outliers=4, device="cuda",
                             extra_pages=[1] * len(lens))
    x = w.q.float()
    x[0, 3] *= 2.0 ** 14            # largest |q| around 2^15.6
    x[0, 9, 17] = 40000.0           # one element above 2^15
    x[1, 7] *= 2.0 ** -12           # largest |q| below 1
    x[2, 10] *= 2.0 ** -40          # tiny row
    x[2, 5] *= 2.0 ** 13            # largest |q| just under 2^15: unscaled
    w = dataclasses.replace(w, q=x.to(torch.bfloat16))
    for kv in (FP8, NVFP4):
        _run(w, kv, g=1.0 if kv != NVFP4 else 0.37, num_sms=37)


def test_tm_matches_mma_kernel(qkvp):
    w = synth.build_workload("both_tm", [777, 64, 3000], heads=32, pool_pages=64, seed=5, outliers=4, device="cuda")
    pools = gpu_pools(w, FP8)
    a, _, _ = gpu_decode(w, FP8, pools, algo=TM)
    b, _, _ = gpu_decode(w, FP8, pools, algo=q.ALGO_MMA_SYNC)
    d = (a.float() - b.float()).abs().max().item()
    assert d < 0.25, d            # both within tolerance of the oracle; they differ by rounding only


def _with_heads(w, heads):
    return dataclasses.replace(w, q=w.q[:, :heads, :].contiguous(), heads=heads)


def _sample_pairs(w, n, seed):
    rng = np.random.default_rng(seed)
    return np.stack([rng.integers(0, w.batch, n), rng.integers(0, w.heads, n)], 1).astype(np.int32)


def _full(name, kv, heads, n_pairs=None, g_mode="one", append=False):
    """One full-size decode step at `heads` heads (the benchmark's heads-sweep configuration): every
    (request, head) output against the oracle, or `n_pairs` sampled ones."""
    w = _with_heads(synth.workload(name, device="cuda"), heads)
    g = 1.0
    if g_mode == "calibrated":
        amax = float(w.src_fp8.view(torch.float8_e4m3fn).float().abs().max())
        g = float(np.float32(amax) / np.float32(2688.0))
    pools = gpu_pools(w, kv, g)
    host = oracle_pools(w, kv, g)
    lens = w.kv_len
    if append:
        src, slots = synth.append_tokens(w, "cuda")
        q.kv_append_quant(src, q.SRC_FP8_E4M3, slots, pools[0], pools[1], kv, g)
        oracle.append(src.cpu().numpy(), oracle.SRC_FP8, slots.cpu().numpy(), kv, g, 64, w.num_pages,
                      host[0].reshape(-1, 288) if kv == NVFP4 else host[0].reshape(-1, 576),
                      host[1].reshape(-1, 36) if kv == NVFP4 else None)
        lens = w.kv_len + 1
    min_splits = 148 if w.batch == 1 else 0
    out, lse, plan = gpu_decode(w, kv, pools, g, min_splits=min_splits, lens=lens, algo=TM)
    assert plan.algo == TM
    pairs = _sample_pairs(w, n_pairs, 7) if n_pairs else np.array(
        [[r, h] for r in range(w.batch) for h in range(w.heads)], np.int32)
    o_ref, lse_ref = oracle_decode(w, kv, host, g, pairs=pairs, lens=lens)
    got = out.float().cpu().numpy()[pairs[:, 0], pairs[:, 1]]
    gl = lse.cpu().numpy()[pairs[:, 0], pairs[:, 1]]
    print(name, heads, compare(got, gl, o_ref, lse_ref), plan.num_segments)
    return plan


@pytest.mark.parametrize("heads", [16, 32, 64])
def test_tm_full_fp8_b44_l32k(qkvp, heads):
    _full("mla_fp8_b44_h128_l32k", FP8, heads)


def test_tm_full_fp8_per_token_b44_l32k(qkvp):
    _full("mla_fp8_b44_h128_l32k", FP8PT, 16, n_pairs=16)


@pytest.mark.parametrize("heads", [16, 32])
def test_tm_full_nvfp4_b10_l160k_with_append(qkvp, heads):
    _full("mla_nvfp4_b10_h128_l160k", NVFP4, heads, n_pairs=8, append=True)


@pytest.mark.parametrize("g_mode", ["one", "calibrated"])
def test_tm_full_nvfp4_b1_l1m(qkvp, g_mode):
    plan = _full("mla_nvfp4_b1_h128_l1m", NVFP4, 16, n_pairs=6, g_mode=g_mode)
    assert plan.num_segments >= 148


def test_tm_full_mixed_pool(qkvp):
    _full("mla_fp8_mixed_b64_h128_pool495552", FP8, 64, n_pairs=32)
