"""The tcgen05 (TMEM, CTA-pair) decode kernel against the FP64 oracle: ragged batches split over
different SM counts, every pool dtype, forced rescales of the running maximum, and the full-size
workloads in the launch configuration the benchmark times: every (request, head) output of the
headline and mixed-batch steps, sampled pairs of the others."""
import dataclasses

import numpy as np
import pytest
import torch

import quantized_kv_paged_gb300 as q
import synth
from tests.helpers import compare, gpu_decode, gpu_pools, oracle_decode, oracle_pools
from tests.test_gpu_decode import _full_check

pytestmark = pytest.mark.gpu

FP8, NVFP4, BF16, FP8PT = q.KV_FP8_E4M3, q.KV_NVFP4, q.KV_BF16, q.KV_FP8_PER_TOKEN
TC = q.ALGO_TCGEN05


def _run(w, kv, g=1.0, raw=False, **kw):
    out, lse, plan = gpu_decode(w, kv, gpu_pools(w, kv, g), g, algo=TC, **kw)
    o_ref, lse_ref = oracle_decode(w, kv, oracle_pools(w, kv, g), g, lens=kw.get("lens"))
    stats = compare(out.float().cpu().numpy().reshape(-1, 512), lse.cpu().numpy().reshape(-1),
                    o_ref, lse_ref, raw=raw)
    return stats, plan


@pytest.mark.parametrize("kv", [FP8, NVFP4, BF16, FP8PT])
def test_tc_ragged_batch_many_splits(qkvp, kv):
    lens = [1, 63, 64, 65, 200, 0, 1000, 4097, 129]
    w = synth.build_workload("ragged", lens, heads=128, pool_pages=180, seed=40 + kv, outliers=4,
                             device="cuda", extra_pages=[1] * len(lens))
    for sms in (4, 37, 152):
        stats, plan = _run(w, kv, g=1.0 if kv != NVFP4 else 0.37, num_sms=sms)
        assert plan.algo == TC and plan.ctas_per_worker == 2


@pytest.mark.parametrize("heads", [16, 64, 96])
def test_tc_fewer_heads_ride_as_zero_rows(qkvp, heads):
    lens = [1, 65, 200, 0, 1000, 4097]
    w = synth.build_workload("few", lens, heads=heads, pool_pages=120, seed=heads, outliers=4, device="cuda",
                             extra_pages=[1] * len(lens))
    for kv in (FP8, NVFP4):
        stats, plan = _run(w, kv, g=1.0 if kv != NVFP4 else 0.37, num_sms=37)
        assert plan.algo == TC


@pytest.mark.parametrize("algo", [TC, q.ALGO_MMA_SYNC])
def test_q_rows_outside_the_unscaled_fp16_range(qkvp, algo):
    """Rows holding a value of 2^15 or more (the whole row, or one element) are rescaled before the
    FP16 conversion; rows whose values sit below 1 or at 2^-40, and a row just under 2^15, are not.
    Both kernels, against the FP64 oracle."""
    lens = [300, 64, 1000]
    w = synth.build_workload("qrange", lens, heads=128, pool_pages=40, seed=11, outliers=4, device="cuda",
                             extra_pages=[1] * len(lens))
    x = w.q.float()
    x[0, 3] *= 2.0 ** 14            # largest |q| around 2^15.6
    x[0, 9, 17] = 40000.0           # one element above 2^15
    x[1, 77] *= 2.0 ** -12          # largest |q| below 1
    x[2, 100] *= 2.0 ** -40         # tiny row
    x[2, 5] *= 2.0 ** 13            # largest |q| just under 2^15: unscaled
    w = dataclasses.replace(w, q=x.to(torch.bfloat16))
    for kv in (FP8, NVFP4):
        g = 1.0 if kv != NVFP4 else 0.37
        out, lse, plan = gpu_decode(w, kv, gpu_pools(w, kv, g), g, algo=algo, num_sms=37)
        o_ref, lse_ref = oracle_decode(w, kv, oracle_pools(w, kv, g), g)
        compare(out.float().cpu().numpy().reshape(-1, 512), lse.cpu().numpy().reshape(-1), o_ref, lse_ref)
        assert plan.algo == algo


def test_tc_tiny_single_page(qkvp):
    w = synth.build_workload("one", [17], heads=128, pool_pages=3, seed=3, device="cuda")
    _run(w, FP8, raw=True, num_sms=2)


def test_tc_long_single_request_min_splits(qkvp):
    w = synth.build_workload("long", [64 * 300 + 5], heads=128, pool_pages=320, seed=1, outliers=4,
                             device="cuda")
    stats, plan = _run(w, NVFP4, g=0.5, num_sms=16, min_splits=40)
    assert plan.num_segments >= 40


def test_tc_lazy_rescale_of_running_max(qkvp):
    """A late token whose logit jumps far above the running maximum forces O to be rescaled."""
    w = synth.build_workload("rescale", [64 * 12, 64 * 5 + 3], heads=128, pool_pages=20, seed=9,
                             device="cuda")
    flat = w.pool_fp8.view(-1, 576)
    for r, tok in ((0, 64 * 9 + 7), (1, 64 * 4 + 1), (0, 64 * 11 + 63)):
        slot = int(w.kv_indices[w.kv_indptr[r] + tok // 64]) * 64 + tok % 64
        # 448 in one nope channel of each CTA's half and in a rope channel: the logit moves by tens,
        # far past the 2^8 (base 2) that triggers a rescale
        for ch in (3, 300, 560):
            flat[slot, ch] = 0x7E
    stats, plan = _run(w, FP8, num_sms=2)        # one segment per request: long runs of pages
    stats, plan = _run(w, FP8, num_sms=8)


def test_tc_matches_mma_kernel(qkvp):
    w = synth.build_workload("both", [777, 64, 3000], heads=128, pool_pages=64, seed=5, outliers=4,
                             device="cuda")
    pools = gpu_pools(w, FP8)
    a, la, _ = gpu_decode(w, FP8, pools, algo=TC)
    b, lb, _ = gpu_decode(w, FP8, pools, algo=q.ALGO_MMA_SYNC)
    d = (a.float() - b.float()).abs().max().item()
    assert d < 0.25, d            # both within tolerance of the oracle; they differ by rounding only


def test_tc_full_fp8_b44_l32k(qkvp):
    """The benchmark's headline step in its launch configuration: every one of the 44 x 128 outputs
    against the FP64 oracle (about a minute of host time)."""
    _full_check("mla_fp8_b44_h128_l32k", FP8, algo=TC, n_pairs=None)


def test_tc_full_fp8_per_token_b44_l32k(qkvp):
    _full_check("mla_fp8_b44_h128_l32k", FP8PT, algo=TC)


def test_tc_full_nvfp4_b10_l160k_with_append(qkvp):
    _full_check("mla_nvfp4_b10_h128_l160k", NVFP4, append=True, n_pairs=8, algo=TC)


@pytest.mark.parametrize("g_mode", ["one", "calibrated"])
def test_tc_full_nvfp4_b1_l1m(qkvp, g_mode):
    plan = _full_check("mla_nvfp4_b1_h128_l1m", NVFP4, g_mode=g_mode, n_pairs=6, algo=TC)
    assert plan.num_segments >= 148


@pytest.mark.parametrize("kv", [FP8, BF16])
def test_tc_full_mixed_pool(qkvp, kv):
    # the fused FP8 decode of the mixed batch: every (request, head) output
    _full_check("mla_fp8_mixed_b64_h128_pool495552", kv, n_pairs=None if kv == FP8 else 16, algo=TC)
