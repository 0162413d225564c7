"""CUDA graphs: mla_decode_run only launches kernels, so a decode step planned outside capture can be
captured and replayed; mla_decode_plan refuses to upload its table during capture (a replay would
read host memory the call no longer owns)."""
import pytest
import torch

import quantized_kv_paged_gb300 as q
import synth
from tests.helpers import gpu_pools

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("algo", [q.ALGO_MMA_SYNC, q.ALGO_TCGEN05, q.ALGO_TCGEN05_TOKENS])
@pytest.mark.parametrize("kv", [q.KV_FP8_E4M3, q.KV_NVFP4])
def test_captured_decode_replays_bit_identical(qkvp, algo, kv):
    w = synth.build_workload("graph", [700, 64, 1300, 5], heads=64, pool_pages=40, seed=31, outliers=2,
                             device="cuda")
    g = 1.0 if kv == q.KV_FP8_E4M3 else 0.5
    pools = gpu_pools(w, kv, g)
    idx = torch.from_numpy(w.kv_indices).cuda()
    p = q.mla_decode_plan(w.kv_indptr, w.kv_len, w.heads, kv, num_sms=37, algo=algo)
    ws = torch.empty(max(p.workspace_bytes, 256), dtype=torch.uint8, device="cuda")
    p = q.mla_decode_plan(w.kv_indptr, w.kv_len, w.heads, kv, num_sms=37, algo=algo, workspace=ws)
    out = torch.empty((w.batch, w.heads, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.batch, w.heads), dtype=torch.float32, device="cuda")

    def step():
        q.mla_decode_run(p, w.q, pools[0], pools[1], w.num_pages, idx, w.sm_scale, g, out, lse, ws)

    step()                                   # eager: the reference bits (and one-time kernel set-up)
    torch.cuda.synchronize()
    ref_out, ref_lse = out.clone(), lse.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
        st = q.mla_decode_plan(w.kv_indptr, w.kv_len, w.heads, kv, num_sms=37, algo=algo, workspace=ws,
                               raise_on_error=False).status
    assert st == q.QKVP_E_UNSUPPORTED
    for _ in range(3):
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
    assert int(ws[p.status_offset:p.status_offset + 4].view(torch.int32).item()) == 0
