"""mla_decode_noalloc: decode for callers that cannot allocate device memory (a serving loop whose
free memory is all in a pre-sized KV pool, or a latency-critical step that must not risk an
allocation's device-wide synchronisation). Its scratch is a fixed array inside the library. It uses
the planner of mla_decode_plan and the same kernel family, so its results must equal the ordinary
plan + run entry points bit for bit, call after call, since each call reuses the array the previous
one left behind; they are also held to the FP64 oracle. Collected last on purpose: a failure here
leaves the rest of the suite already run."""
import numpy as np
import pytest
import torch

import quantized_kv_paged_gb300 as q
import synth
from tests.helpers import compare, gpu_decode, gpu_pools, oracle_decode, oracle_pools


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
        # the same kernel family and SM count as the no-allocation call: the same split, so the same bits
        ref_out, ref_lse, plan = gpu_decode(w, kv, pools, g, num_sms=sms, algo=q.ALGO_MMA_SYNC)
        assert plan.num_split_requests > 0        # the scratch partials are exercised
        out, lse = _noalloc(w, kv, pools, g, sms)
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
        o_ref, l_ref = oracle_decode(w, kv, oracle_pools(w, kv, g), g)
        compare(out.float().cpu().numpy().reshape(-1, 512), lse.cpu().numpy().reshape(-1), o_ref, l_ref)


@pytest.mark.gpu
def test_noalloc_is_refused_during_stream_capture(cuda_device):
    """A captured graph would replay a host table that later calls overwrite: the call refuses."""
    q.load()
    w = synth.build_workload("noalloc_cap", [300], heads=16, pool_pages=8, seed=3, device="cuda")
    out = torch.empty((1, 16, 512), dtype=torch.bfloat16, device="cuda")
    idx = torch.from_numpy(w.kv_indices).cuda()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        st = q.mla_decode_noalloc(w.kv_indptr, w.kv_len, 16, q.KV_FP8_E4M3, w.q, w.pool_fp8, None, w.num_pages,
                                  idx, w.sm_scale, 1.0, out, None, num_sms=8, raise_on_error=False)
    assert st == q.QKVP_E_UNSUPPORTED


def test_noalloc_rejects_problems_beyond_the_scratch():
    L = q.load()
    # 300 split partials x 128 heads x 512 x 4 bytes > 64 MiB: refused before any device work
    lens = np.array([1 << 20], np.int32)
    ptr = np.array([0, 16384], np.int32)
    st = L.mla_decode_noalloc(ptr.ctypes.data, lens.ctypes.data, 1, 128, q.KV_FP8_E4M3, 152, 300,
                              16, 16, None, 16384, 16, 0.1, 1.0, 16, None, None)
    assert st == q.QKVP_E_WORKSPACE
    big, big_ptr = np.zeros(9000, np.int32), np.zeros(9001, np.int32)
    st = L.mla_decode_noalloc(big_ptr.ctypes.data, big.ctypes.data, 9000, 128,
                              q.KV_FP8_E4M3, 152, 0, 16, 16, None, 1, 16, 0.1, 1.0, 16, None, None)
    assert st == q.QKVP_E_WORKSPACE
