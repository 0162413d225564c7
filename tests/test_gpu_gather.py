"""The extend-path gather into an FP8 workspace and the gather-then-cast baseline: the CUDA path
through the C ABI against the oracle, byte for byte, on ragged and full-size workloads."""
import numpy as np
import pytest
import torch

import oracle
import quantized_kv_paged_gb300 as q
import synth
from tests.helpers import gpu_pools, oracle_pools

pytestmark = pytest.mark.gpu


def _tables(w, lens=None, dev="cuda"):
    lens = w.kv_len if lens is None else np.asarray(lens)
    tok = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    return (torch.from_numpy(w.kv_indptr.astype(np.int32)).to(dev), torch.from_numpy(w.kv_indices).to(dev),
            torch.from_numpy(tok).to(dev), tok)


def _gather_gpu(pools, kv, g, w, lens=None, indices=None):
    ip, ix, tk, tok = _tables(w, lens)
    if indices is not None:
        ix = torch.from_numpy(indices).cuda()
    out = torch.full((int(tok[-1]), 576), 0xA5, dtype=torch.uint8, device="cuda")
    q.kv_gather_fp8(pools[0], pools[1], kv, g, ip, ix, tk, out, num_pages=w.num_pages)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("kv,g", [(q.KV_FP8_E4M3, 1.0), (q.KV_NVFP4, 1.0), (q.KV_NVFP4, 0.37), (q.KV_NVFP4, 2.0 ** -6)])
def test_gather_ragged_matches_oracle_bytes(qkvp, kv, g):
    lens = [1, 63, 64, 65, 200, 0, 1000, 4097, 129]
    w = synth.build_workload("ragged", lens, heads=16, pool_pages=180, seed=11, outliers=4, device="cuda",
                             extra_pages=[1] * len(lens))
    got = _gather_gpu(gpu_pools(w, kv, g), kv, g, w)
    host = oracle_pools(w, kv, g)
    tok = np.concatenate([[0], np.cumsum(lens)])
    ref, bad = oracle.gather_fp8(host[0], host[1], kv, g, 64, w.num_pages, w.kv_indptr, w.kv_indices, tok)
    assert bad == 0
    assert np.array_equal(got, ref)


def test_gather_bad_page_ids_give_zero_rows(qkvp):
    w = synth.build_workload("bad", [130, 70], heads=16, pool_pages=6, seed=4, device="cuda")
    idx = w.kv_indices.copy()
    idx[1] = 1 << 30                     # second page of request 0 lies outside the pool
    idx[2] = -3
    got = _gather_gpu(gpu_pools(w, q.KV_NVFP4, 1.0), q.KV_NVFP4, 1.0, w, indices=idx)
    host = oracle_pools(w, q.KV_NVFP4, 1.0)
    ref, bad = oracle.gather_fp8(host[0], host[1], q.KV_NVFP4, 1.0, 64, w.num_pages, w.kv_indptr, idx,
                                 np.array([0, 130, 200]))
    assert bad == 64 + 2 and np.array_equal(got, ref)   # tokens 64..127 and 128..129 of request 0
    assert np.all(got[64:128] == 0)


def test_gather_full_size_nvfp4_extend_workload(qkvp):
    """The NVFP4 10 x 163,840 pool (bulk-filled by the library's append), whole prefixes gathered:
    944 MB of workspace; every byte of sampled rows checked, plus per-row checksums of all rows."""
    w = synth.workload("mla_nvfp4_b10_h128_l160k", device="cuda")
    g = 1.0
    pools = gpu_pools(w, q.KV_NVFP4, g)
    ip, ix, tk, tok = _tables(w)
    out = torch.empty((int(tok[-1]), 576), dtype=torch.uint8, device="cuda")
    q.kv_gather_fp8(pools[0], pools[1], q.KV_NVFP4, g, ip, ix, tk, out, num_pages=w.num_pages)
    torch.cuda.synchronize()
    host = oracle_pools(w, q.KV_NVFP4, g)
    rng = np.random.default_rng(5)
    for r in range(w.batch):
        ts = rng.integers(0, w.kv_len[r], 64)
        # the oracle on a one-page table holding each sampled token's page
        pages = w.kv_indices[w.kv_indptr[r] + ts // 64]
        for t, pg in zip(ts, pages):
            ref, _ = oracle.gather_fp8(host[0], host[1], q.KV_NVFP4, g, 64, w.num_pages, [0, 1], [pg],
                                       [0, 64])
            row = out[int(tok[r] + t)].cpu().numpy()
            assert np.array_equal(row, ref[t % 64]), (r, t)


def test_gather_pages_bf16_matches_oracle(qkvp):
    w = synth.workload("mla_fp8_mixed_b64_h128_pool495552", device="cuda")
    ids = w.kv_indices.copy()
    ids[::97] = w.num_pages + 5          # a few ids outside the pool: zero pages
    ids_d = torch.from_numpy(ids).cuda()
    out = torch.full((ids.size, 64, 576), 0x1234, dtype=torch.int16, device="cuda")
    q.kv_gather_pages_bf16(w.pool_fp8, ids_d, out)
    torch.cuda.synchronize()
    sel = np.random.default_rng(6).integers(0, ids.size, 40)
    sel = np.concatenate([sel, np.arange(0, ids.size, 97)[:5]])
    ref = oracle.gather_pages_bf16(w.pool_fp8.cpu().numpy(), ids[sel])
    got = out.cpu().numpy()[sel].view(np.uint16)
    assert np.array_equal(got, ref)


def test_gather_then_cast_decode_equals_cast_then_attend(qkvp):
    """The compact BF16 pool read through identity page ids decodes exactly as the whole-pool cast
    read through the original page ids (same kernel, same values, same order)."""
    w = synth.build_workload("gtc", [300, 64, 1, 777], heads=128, pool_pages=40, seed=9, outliers=4, device="cuda")
    full = torch.empty((w.num_pages, 64, 576), dtype=torch.int16, device="cuda")
    q.kv_pool_cast_bf16(w.pool_fp8, full)
    compact = torch.empty((w.kv_indices.size, 64, 576), dtype=torch.int16, device="cuda")
    q.kv_gather_pages_bf16(w.pool_fp8, torch.from_numpy(w.kv_indices).cuda(), compact)
    outs = []
    for pool, idx in ((full, w.kv_indices), (compact, np.arange(w.kv_indices.size, dtype=np.int32))):
        plan = q.mla_decode_plan(w.kv_indptr, w.kv_len, w.heads, q.KV_BF16, num_sms=37)
        ws = torch.empty(max(256, plan.workspace_bytes), dtype=torch.uint8, device="cuda")
        plan = q.mla_decode_plan(w.kv_indptr, w.kv_len, w.heads, q.KV_BF16, num_sms=37, workspace=ws)
        o = torch.empty((w.batch, w.heads, 512), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((w.batch, w.heads), dtype=torch.float32, device="cuda")
        q.mla_decode_run(plan, w.q, pool, None, pool.shape[0], torch.from_numpy(idx).cuda(), w.sm_scale, 1.0,
                         o, lse, ws)
        torch.cuda.synchronize()
        outs.append((o.cpu(), lse.cpu()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
