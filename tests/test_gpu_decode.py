"""Decode parity: the CUDA path through the C ABI against the FP64 oracle, element by element on
small and ragged cases, and on sampled (request, head) pairs at the full workload sizes in the
launch configuration the benchmark times."""
import math

import numpy as np
import pytest
import torch

import oracle
import quantized_kv_paged_gb300 as q
import synth
from tests.helpers import compare, gpu_decode, gpu_pools, oracle_decode, oracle_pools

pytestmark = pytest.mark.gpu

FP8, NVFP4, BF16, FP8PT = q.KV_FP8_E4M3, q.KV_NVFP4, q.KV_BF16, q.KV_FP8_PER_TOKEN


def _run(w, kv, g=1.0, raw=False, **kw):
    out, lse, plan = gpu_decode(w, kv, gpu_pools(w, kv, g), g, algo=q.ALGO_MMA_SYNC, **kw)
    o_ref, lse_ref = oracle_decode(w, kv, oracle_pools(w, kv, g), g, lens=kw.get("lens"))
    stats = compare(out.float().cpu().numpy().reshape(-1, 512), lse.cpu().numpy().reshape(-1),
                    o_ref, lse_ref, raw=raw)
    return stats, plan


@pytest.mark.parametrize("kv", [FP8, NVFP4])
def test_tiny_workload(qkvp, kv):
    w = synth.workload("mla_tiny_b1_h16_l256", device="cuda")
    stats, _ = _run(w, kv, raw=True)
    print(stats)


@pytest.mark.parametrize("heads", [16, 32, 48, 64, 128])
@pytest.mark.parametrize("kv", [FP8, NVFP4, BF16, FP8PT])
def test_ragged_batch_many_splits(qkvp, heads, kv):
    lens = [1, 63, 64, 65, 200, 0, 1000, 4097, 129]
    w = synth.build_workload("ragged", lens, heads=heads, pool_pages=180, seed=heads + kv,
                             outliers=4, device="cuda", extra_pages=[1] * len(lens))
    for sms in (4, 37, 152):
        stats, plan = _run(w, kv, g=1.0 if kv != NVFP4 else 0.37, num_sms=sms)
        assert plan.num_empty_requests == 1


def test_min_splits_and_single_request(qkvp):
    w = synth.build_workload("long", [64 * 150 + 13], heads=64, pool_pages=160, seed=1, outliers=4,
                             device="cuda")
    stats, plan = _run(w, NVFP4, g=0.5, num_sms=16, min_splits=40)
    assert plan.num_segments >= 40


def test_all_requests_empty(qkvp):
    w = synth.build_workload("empty", [0, 0], heads=16, pool_pages=2, seed=2, device="cuda",
                             extra_pages=[1, 0])
    out, lse, plan = gpu_decode(w, FP8, gpu_pools(w, FP8), algo=q.ALGO_MMA_SYNC)
    assert torch.all(out == 0) and torch.all(torch.isinf(lse)) and torch.all(lse < 0)


def test_bad_page_ids_are_masked_not_read(qkvp):
    w = synth.build_workload("bad", [130, 70], heads=16, pool_pages=6, seed=4, device="cuda")
    idx = w.kv_indices.copy()
    idx[1] = 1 << 30          # second page of request 0 lies outside the pool
    out, lse, _ = gpu_decode(w, FP8, gpu_pools(w, FP8), indices=idx, algo=q.ALGO_MMA_SYNC)
    assert torch.all(torch.isfinite(out.float()))
    # request 0 then attends only its first page and its last two tokens; request 1 is untouched
    w0 = synth.build_workload("bad", [130, 70], heads=16, pool_pages=6, seed=4, device="cpu")
    o1, l1 = oracle_decode(w0, FP8, oracle_pools(w0, FP8), pairs=np.array([[1, h] for h in range(16)]))
    compare(out[1].float().cpu().numpy(), lse[1].cpu().numpy(), o1, l1, raw=True)


def test_subnormal_latents_survive_dequant(qkvp):
    """E4M3 subnormals (|x| < 2^-6) must dequantize exactly: a pool made only of them."""
    w = synth.build_workload("sub", [256], heads=16, pool_pages=4, seed=5, device="cuda")
    codes = torch.randint(1, 8, (w.num_pages, 64, 576), dtype=torch.uint8, device="cuda")
    sign = torch.randint(0, 2, codes.shape, dtype=torch.uint8, device="cuda") << 7
    w.pool_fp8.copy_(codes | sign)
    out, lse, _ = gpu_decode(w, FP8, (w.pool_fp8, None), algo=q.ALGO_MMA_SYNC)
    o_ref, lse_ref = oracle_decode(w, FP8, (w.pool_fp8.cpu().numpy(), None))
    got = out.float().cpu().numpy().reshape(-1, 512)
    assert np.abs(o_ref).max() > 1e-4
    assert np.allclose(got, o_ref, rtol=1e-2, atol=2e-5), float(np.abs(got - o_ref).max())


def test_nvfp4_scale_folding(qkvp):
    """The global scale enters through the logit scale and the output scale."""
    w = synth.build_workload("g", [300, 77], heads=32, pool_pages=8, seed=6, outliers=2, device="cuda")
    for g in (1.0, 2.0 ** -5, 7.25):
        _run(w, NVFP4, g=g, num_sms=8)


@pytest.mark.parametrize("algo", [q.ALGO_MMA_SYNC, q.ALGO_TCGEN05])
def test_plan_uploads_in_flight(qkvp, algo):
    """Six plans of different lengths are uploaded into six workspaces and decoded with no host
    synchronisation in between, queued behind a few milliseconds of other GPU work, so more table
    uploads are in flight than the library has pinned staging buffers (four). Each result equals the
    same plan decoded with a synchronisation after every call, bit for bit."""
    w = synth.build_workload("flight", [700, 64, 1300, 5, 300], heads=32, pool_pages=60, seed=21, outliers=2,
                             device="cuda", extra_pages=[1] * 5)
    pools = gpu_pools(w, FP8)
    idx = torch.from_numpy(w.kv_indices).to("cuda")
    cases = [np.maximum(w.kv_len - 3 * k, 0).astype(np.int32) for k in range(6)]

    def workspace(lens):
        p = q.mla_decode_plan(w.kv_indptr, lens, w.heads, FP8, num_sms=37, algo=algo)
        return torch.empty(max(p.workspace_bytes, 256), dtype=torch.uint8, device="cuda")

    def decode(lens, ws):
        out = torch.empty((w.batch, w.heads, 512), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((w.batch, w.heads), dtype=torch.float32, device="cuda")
        p = q.mla_decode_plan(w.kv_indptr, lens, w.heads, FP8, num_sms=37, algo=algo, workspace=ws)
        q.mla_decode_run(p, w.q, pools[0], pools[1], w.num_pages, idx, w.sm_scale, 1.0, out, lse, ws)
        return out, lse

    wss = [workspace(lens) for lens in cases]
    ref = []
    for lens, ws in zip(cases, wss):
        ref.append(decode(lens, ws))
        torch.cuda.synchronize()
    a = torch.randn(4096, 4096, device="cuda")
    for _ in range(20):
        a = a @ a / 64.0                       # keeps the stream busy while the uploads queue
    got = [decode(lens, ws) for lens, ws in zip(cases, wss)]
    torch.cuda.synchronize()
    for (o, l), (ro, rl) in zip(got, ref):
        assert torch.equal(o, ro) and torch.equal(l, rl)


# ---- full sizes, bench launch configuration, sampled outputs --------------------------------------

def _sample_pairs(w, n, seed):
    rng = np.random.default_rng(seed)
    r = rng.integers(0, w.batch, n)
    h = rng.integers(0, w.heads, n)
    return np.stack([r, h], 1).astype(np.int32)


def _full_check(name, kv, g_mode="one", n_pairs=12, append=False, algo=0):
    w = synth.workload(name, device="cuda")
    if g_mode == "calibrated":
        amax = float(w.src_fp8.view(torch.float8_e4m3fn).float().abs().max())
        g = float(np.float32(amax) / np.float32(2688.0))
    else:
        g = 1.0
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
    if kv == NVFP4:
        assert np.array_equal(pools[0].cpu().numpy(), host[0]) and np.array_equal(pools[1].cpu().numpy(), host[1])
    if kv == FP8PT:
        assert np.array_equal(pools[0].cpu().numpy(), host[0])
    min_splits = 148 if w.batch == 1 else 0
    out, lse, plan = gpu_decode(w, kv, pools, g, min_splits=min_splits, lens=lens, algo=algo)
    assert torch.all(torch.isfinite(out.float())) and torch.all(torch.isfinite(lse))
    # n_pairs None: every (request, head) output of the step
    pairs = _sample_pairs(w, n_pairs, 7) if n_pairs else np.array(
        [[r, h] for r in range(w.batch) for h in range(w.heads)], np.int32)
    o_ref, lse_ref = oracle_decode(w, kv, host, g, pairs=pairs, lens=lens)
    got = out.float().cpu().numpy()[pairs[:, 0], pairs[:, 1]]
    gl = lse.cpu().numpy()[pairs[:, 0], pairs[:, 1]]
    stats = compare(got, gl, o_ref, lse_ref)
    print(name, stats, plan.num_segments)
    return plan


def test_full_fp8_b44_l32k(qkvp):
    _full_check("mla_fp8_b44_h128_l32k", FP8, algo=q.ALGO_MMA_SYNC)


def test_full_fp8_per_token_b44_l32k(qkvp):
    _full_check("mla_fp8_b44_h128_l32k", FP8PT, algo=q.ALGO_MMA_SYNC)


def test_full_nvfp4_b10_l160k_with_append(qkvp):
    _full_check("mla_nvfp4_b10_h128_l160k", NVFP4, append=True, n_pairs=8, algo=q.ALGO_MMA_SYNC)


@pytest.mark.parametrize("g_mode", ["one", "calibrated"])
def test_full_nvfp4_b1_l1m(qkvp, g_mode):
    plan = _full_check("mla_nvfp4_b1_h128_l1m", NVFP4, g_mode=g_mode, n_pairs=6, algo=q.ALGO_MMA_SYNC)
    assert plan.num_segments >= 148


@pytest.mark.parametrize("kv", [FP8, BF16])
def test_full_mixed_pool(qkvp, kv):
    _full_check("mla_fp8_mixed_b64_h128_pool495552", kv, n_pairs=16, algo=q.ALGO_MMA_SYNC)


# ---- FP8 Q.K^T (QKVP_ALGO_MMA_FP8): two-term E4M3 Q against the page's E4M3 bytes -------------------

F8QK = q.ALGO_MMA_FP8


@pytest.mark.parametrize("heads", [16, 32, 48, 128])
@pytest.mark.parametrize("kv", [FP8, FP8PT])
def test_fp8_qk_ragged_batch(qkvp, heads, kv):
    """The FP8 Q.K^T variant meets the same tolerance against the FP64 oracle as the FP16 kernels, on
    ragged batches with x20 outlier channels, empty requests and split requests."""
    lens = [1, 63, 64, 65, 200, 0, 1000, 4097, 129]
    w = synth.build_workload("ragged_f8", lens, heads=heads, pool_pages=180, seed=70 + heads + kv,
                             outliers=4, device="cuda", extra_pages=[1] * len(lens))
    for sms in (4, 37, 152):
        out, lse, plan = gpu_decode(w, kv, gpu_pools(w, kv), algo=F8QK, num_sms=sms)
        assert plan.algo == F8QK and plan.ctas_per_worker == heads // (32 if heads % 32 == 0 else 16)
        o_ref, lse_ref = oracle_decode(w, kv, oracle_pools(w, kv))
        compare(out.float().cpu().numpy().reshape(-1, 512), lse.cpu().numpy().reshape(-1), o_ref, lse_ref)


def test_fp8_qk_q_rows_of_any_magnitude(qkvp):
    """Each head row gets its own power-of-two scale into the E4M3 range: rows at 2^15, one element of
    40,000, rows below 1 and at 2^-40 all meet the tolerance."""
    import dataclasses
    w = synth.build_workload("qrange_f8", [300, 64, 1000], heads=32, pool_pages=40, seed=12, outliers=4,
                             device="cuda", extra_pages=[1] * 3)
    x = w.q.float()
    x[0, 3] *= 2.0 ** 14
    x[0, 9, 17] = 40000.0
    x[1, 7] *= 2.0 ** -12
    x[2, 10] *= 2.0 ** -40
    w = dataclasses.replace(w, q=x.to(torch.bfloat16))
    out, lse, _ = gpu_decode(w, FP8, gpu_pools(w, FP8), algo=F8QK, num_sms=37)
    o_ref, lse_ref = oracle_decode(w, FP8, oracle_pools(w, FP8))
    compare(out.float().cpu().numpy().reshape(-1, 512), lse.cpu().numpy().reshape(-1), o_ref, lse_ref)


def test_full_fp8_b44_l32k_fp8_qk(qkvp):
    _full_check("mla_fp8_b44_h128_l32k", FP8, algo=F8QK)
