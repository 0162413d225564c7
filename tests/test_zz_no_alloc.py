"""mla_decode_noalloc: decode for callers that cannot allocate device memory (a serving loop whose
free memory is all in a pre-sized KV pool, or a latency-critical step that must not risk an
allocation's device-wide synchronisation). Its scratch is a fixed array inside the library; its
results must match the ordinary plan + run entry points, call after call, since each call reuses
the array the previous one left behind. Collected last on purpose: a failure here leaves the rest
of the suite already run."""
import numpy as np
import pytest
import torch

import quantized_kv_paged_gb300 as q
import synth
from tests.helpers import compare, gpu_decode, gpu_pools


def _noalloc(w, kv, pools, g, num_sms):
    out = torch.full((w.batch, w.heads, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((w.batch, w.heads), float("nan"), dtype=torch.float32, device="cuda")
    idx = torch.from_numpy(w.kv_indices).cuda()
    q.mla_decode_noalloc(w.kv_indptr, w.kv_len, w.heads, kv, w.q, pools[0], pools[1], w.num_pages, idx,
                         w.sm_scale, g, out, lse, num_sms=num_sms)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.gpu
def test_noalloc_matches_plan_and_run_two_calls_in_a_row(cuda_device):
    q.load()
    cases = [
        # (lengths, heads, kv dtype, global scale, SMs): the second call is smaller than the first, so
        # it runs on scratch that still holds the first call's table and partials
        ([1000, 1, 0, 4097, 65, 300], 128, q.KV_NVFP4, 0.25, 37),
        ([256, 70], 32, q.KV_FP8_E4M3, 1.0, 16),
    ]
    for lens, heads, kv, g, sms in cases:
        w = synth.build_workload("noalloc", lens, heads=heads, pool_pages=200, seed=heads + len(lens),
                                 outliers=4, device="cuda")
        pools = gpu_pools(w, kv, g)
        # the same kernel family as the no-allocation call, so both plans split the work alike
        ref_out, ref_lse, plan = gpu_decode(w, kv, pools, g, num_sms=sms, algo=q.ALGO_MMA_SYNC)
        assert plan.num_split_requests > 0        # the scratch partials are exercised
        out, lse = _noalloc(w, kv, pools, g, sms)
        compare(out.float().cpu().numpy().reshape(-1, 512), lse.cpu().numpy().reshape(-1),
                ref_out.double().cpu().numpy().reshape(-1, 512), ref_lse.double().cpu().numpy().reshape(-1))


def test_noalloc_rejects_problems_beyond_the_scratch():
    q.load()
    L = q.load()
    # 300 split partials x 128 heads x 512 x 4 bytes > 64 MiB: refused before any device work
    lens = np.array([1 << 20], np.int32)
    ptr = np.array([0, 16384], np.int32)
    st = L.mla_decode_noalloc(ptr.ctypes.data, lens.ctypes.data, 1, 128, q.KV_FP8_E4M3, 152, 300,
                              16, 16, None, 16384, 16, 0.1, 1.0, 16, None, None)
    assert st == q.QKVP_E_WORKSPACE
    big = np.zeros(9000, np.int32)
    st = L.mla_decode_noalloc(np.zeros(9001, np.int32).ctypes.data, big.ctypes.data, 9000, 128,
                              q.KV_FP8_E4M3, 152, 0, 16, 16, None, 1, 16, 0.1, 1.0, 16, None, None)
    assert st == q.QKVP_E_WORKSPACE
