"""The C ABI without a GPU: the library loads and exports every function qkvp.h declares; argument
checks fail before any launch; the planner's split is balanced and honours min_splits."""
import ctypes
import os
import re

import numpy as np
import pytest

import quantized_kv_paged_gb300 as q
from tests.conftest import ROOT


@pytest.fixture(scope="module")
def lib():
    from quantized_kv_paged_gb300 import build
    build.build()
    return q.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "qkvp.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|const char\*)\s+(\w+)\s*\(", src, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert set(q.EXPORTS) == set(names)
    for n in names:
        assert hasattr(lib, n), n
        assert ctypes.cast(getattr(lib, n), ctypes.c_void_p).value


def test_status_strings(lib):
    assert q.status_string(0) == "ok"
    for s in (-1, -2, -3, -4, 7):
        assert q.status_string(s)
    assert q.qkvp_version() >= 100


def plan(indptr, lens, heads=128, kv=q.KV_FP8_E4M3, sms=152, min_splits=0, algo=0, page_size=64):
    return q.mla_decode_plan(indptr, lens, heads, kv, num_sms=sms, min_splits=min_splits,
                             algo=algo, page_size=page_size, raise_on_error=False)


def test_plan_rejects_bad_arguments(lib):
    ok_ptr, ok_len = np.array([0, 2], np.int32), np.array([100], np.int32)
    assert plan(ok_ptr, ok_len).status == q.QKVP_OK
    assert plan(ok_ptr, ok_len, page_size=32).status == q.QKVP_E_UNSUPPORTED
    for h in (8, 24 + 1, 144, 0):
        assert plan(ok_ptr, ok_len, heads=h).status == q.QKVP_E_UNSUPPORTED
    assert plan(ok_ptr, ok_len, kv=9).status == q.QKVP_E_UNSUPPORTED
    assert plan(ok_ptr, ok_len, kv=q.KV_FP8_PER_TOKEN).status == q.QKVP_OK
    assert plan(np.array([1, 3], np.int32), ok_len).status == q.QKVP_E_INVALID       # indptr[0] != 0
    assert plan(np.array([0, 1], np.int32), ok_len).status == q.QKVP_E_INVALID       # 100 tokens, 1 page
    assert plan(np.array([0, 2], np.int32), np.array([-1], np.int32)).status == q.QKVP_E_INVALID
    assert plan(np.array([0, 2, 1], np.int32), np.array([5, 5], np.int32)).status == q.QKVP_E_INVALID
    assert plan(ok_ptr, ok_len, min_splits=-1).status == q.QKVP_E_INVALID
    assert plan(ok_ptr, ok_len, algo=7).status == q.QKVP_E_UNSUPPORTED
    # AUTO: quantized pools take the token-major kernel at 32-64 heads, mma.sync at 16, the tcgen05
    # CTA-pair kernel above 64; BF16 pools mma.sync below 64 heads, the CTA-pair kernel from 64
    for kv in (q.KV_FP8_E4M3, q.KV_NVFP4, q.KV_FP8_PER_TOKEN):
        assert plan(ok_ptr, ok_len, heads=16, kv=kv).algo == q.ALGO_MMA_SYNC
        for heads in (32, 48, 64):
            assert plan(ok_ptr, ok_len, heads=heads, kv=kv).algo == q.ALGO_TCGEN05_TOKENS
        for heads in (80, 128):
            assert plan(ok_ptr, ok_len, heads=heads, kv=kv).algo == q.ALGO_TCGEN05
    for heads in (16, 32, 48):
        assert plan(ok_ptr, ok_len, heads=heads, kv=q.KV_BF16).algo == q.ALGO_MMA_SYNC
    assert plan(ok_ptr, ok_len, heads=64, kv=q.KV_BF16).algo == q.ALGO_TCGEN05
    assert plan(ok_ptr, ok_len, heads=16, algo=q.ALGO_TCGEN05).status == q.QKVP_OK


def test_plan_workspace_too_small_reports_size(lib):
    ptr, lens = np.array([0, 512, 1024], np.int32), np.array([32768, 32768], np.int32)
    p = plan(ptr, lens)
    st = lib.mla_decode_plan(ptr.ctypes.data, lens.ctypes.data, 2, 128, 64, 1, 152, 0, 0,
                             ctypes.c_void_p(256), 64, None, ctypes.byref(p))
    assert st == q.QKVP_E_WORKSPACE and p.workspace_bytes > 64


def test_split_is_balanced_and_covers_every_page(lib):
    lens = np.array([32768] * 44, np.int32)
    ptr = np.concatenate([[0], np.cumsum((lens + 63) // 64)]).astype(np.int32)
    p = plan(ptr, lens, algo=q.ALGO_MMA_SYNC)   # 76 workers of two 64-head CTAs, equal page quotas
    assert p.total_pages == 44 * 512 and p.total_tokens == 44 * 32768
    assert p.ctas_per_worker * p.num_workers <= 152
    # makespan is the ceiling of the mean: no worker holds more than one page above it
    assert p.max_worker_pages == -(-p.total_pages // p.num_workers)
    assert p.min_worker_pages >= p.total_pages - (p.num_workers - 1) * p.max_worker_pages
    assert p.num_segments >= 44 and p.workspace_bytes >= p.num_partials * 128 * 512 * 4
    # a request's 512 contiguous pages meet at most ceil(512 / quota) + 1 worker ranges
    assert 2 <= p.max_request_segments <= -(-512 // p.max_worker_pages) + 1
    assert p.num_wide_requests == 0   # every request merges in the narrow combine CTAs


def test_min_splits_spreads_one_long_request(lib):
    lens = np.array([1 << 20], np.int32)
    ptr = np.array([0, 16384], np.int32)
    p = plan(ptr, lens, min_splits=148)
    assert p.num_segments >= 148 and p.num_split_requests == 1 and p.num_partials == p.num_segments
    assert p.max_request_segments == p.num_segments and p.num_wide_requests == 1
    p0 = plan(ptr, lens, min_splits=0)
    assert p0.num_segments == p0.num_workers == p0.max_request_segments


def test_ragged_and_empty_requests(lib):
    lens = np.array([0, 1, 64, 65, 0, 1000], np.int32)
    ptr = np.concatenate([[0], np.cumsum((lens + 63) // 64 + 1)]).astype(np.int32)   # 1 spare page each
    p = plan(ptr, lens, heads=16, sms=4)
    assert p.num_empty_requests == 2
    assert p.total_pages == sum((int(l) + 63) // 64 for l in lens)
    assert p.num_workers == 4 and p.ctas_per_worker == 1
    assert (p.max_request_segments >= 2) == (p.num_split_requests > 0)
    assert p.max_request_segments <= p.num_segments
    assert (p.num_wide_requests > 0) == (p.max_request_segments > 8)
    # one worker per 16-head CTA group at 16 heads: with 4 workers no request meets more than 4
    assert p.num_wide_requests == 0
    pw = plan(ptr, lens, heads=16, sms=152)
    assert pw.max_request_segments > 8 and 1 <= pw.num_wide_requests <= 2


def test_run_and_append_reject_before_launch(lib):
    p = plan(np.array([0, 2], np.int32), np.array([100], np.int32))
    # a size-only plan carries no upload: run refuses it
    st = lib.mla_decode_run(ctypes.byref(p), 16, 16, None, 10, 16, 0.1, 1.0, 16, None, 256,
                            1 << 30, None)
    assert st == q.QKVP_E_INVALID
    f = lib.kv_append_quant
    assert f(16, 1, 4, 16, 16, 16, 1, 1.0, 64, 10, None) == q.QKVP_E_INVALID      # FP8 with scale pool
    assert f(16, 1, 4, 16, 16, None, 1, 2.0, 64, 10, None) == q.QKVP_E_INVALID    # FP8 with g != 1
    assert f(16, 1, 4, 16, 16, None, 2, 1.0, 64, 10, None) == q.QKVP_E_INVALID    # NVFP4 without scales
    assert f(16, 1, 4, 16, 16, 16, 2, 0.0, 64, 10, None) == q.QKVP_E_INVALID      # g = 0
    assert f(16, 1, 4, 16, 16, 16, 2, float("nan"), 64, 10, None) == q.QKVP_E_INVALID
    assert f(16, 1, 4, 16, 16, 16, 3, 1.0, 64, 10, None) == q.QKVP_E_UNSUPPORTED  # BF16 pool
    assert f(16, 1, 4, 16, 16, 16, 4, 1.0, 64, 10, None) == q.QKVP_E_INVALID      # per-token FP8 + scale pool
    assert f(16, 1, 4, 16, 16, None, 4, 0.5, 64, 10, None) == q.QKVP_E_INVALID    # per-token FP8, g != 1
    assert f(16, 1, 0, 16, 16, None, 4, 1.0, 64, 10, None) == q.QKVP_OK            # accepted, nothing to do
    assert f(16, 1, 4, 16, 16, 16, 2, 1.0, 32, 10, None) == q.QKVP_E_UNSUPPORTED  # page size
    assert f(None, 1, 4, 16, 16, 16, 2, 1.0, 64, 10, None) == q.QKVP_E_INVALID
    assert f(17, 1, 4, 16, 16, 16, 2, 1.0, 64, 10, None) == q.QKVP_E_INVALID      # misaligned source
    assert f(16, 1, -1, 16, 16, 16, 2, 1.0, 64, 10, None) == q.QKVP_E_INVALID
    assert f(16, 1, 0, 16, 16, 16, 2, 1.0, 64, 10, None) == q.QKVP_OK              # nothing to do
    # a plan with a valid header but an output that is only 4-byte aligned: refused before launch
    # (the attend kernels store 16-byte vectors)
    pv = plan(np.array([0, 2], np.int32), np.array([100], np.int32))
    pv.magic = 0x716B76702D706C31
    st = lib.mla_decode_attend(ctypes.byref(pv), 16, 16, None, 10, 16, 0.1, 1.0, 0x1004, None, 256,
                               pv.workspace_bytes, None)
    assert st == q.QKVP_E_INVALID
    # a pool that is 16- but not 32-byte aligned (the attend kernels use 32-byte loads)
    st = lib.mla_decode_attend(ctypes.byref(pv), 16, 0x1010, None, 10, 16, 0.1, 1.0, 0x1000, None, 256,
                               pv.workspace_bytes, None)
    assert st == q.QKVP_E_INVALID
    assert lib.kv_pool_cast_bf16(16, 17, 16, None) == q.QKVP_E_INVALID
    assert lib.qkvp_encode_f32(16, 4, 3, 16, None) == q.QKVP_E_INVALID


def test_gather_entry_points_reject_before_launch(lib):
    f = lib.kv_gather_fp8
    ok = dict(kv=16, sc=16, dt=2, g=1.0, ps=64, np_=10, ip=16, ix=16, nnz=4, tok=16, b=2, t=100, out=16)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["kv"], a["sc"], a["dt"], a["g"], a["ps"], a["np_"], a["ip"], a["ix"], a["nnz"], a["tok"],
                 a["b"], a["t"], a["out"], None)
    assert call(ps=32) == q.QKVP_E_UNSUPPORTED
    assert call(dt=3) == q.QKVP_E_UNSUPPORTED                 # BF16 pool
    assert call(dt=4, sc=None) == q.QKVP_E_UNSUPPORTED        # per-token-scaled FP8 pool
    assert call(dt=7) == q.QKVP_E_INVALID
    assert call(g=0.0) == q.QKVP_E_INVALID
    assert call(g=float("inf")) == q.QKVP_E_INVALID
    assert call(dt=1) == q.QKVP_E_INVALID                     # FP8 with a scale pool
    assert call(dt=1, sc=None, g=2.0) == q.QKVP_E_INVALID     # FP8 with g != 1
    assert call(sc=None) == q.QKVP_E_INVALID                  # NVFP4 without scales
    assert call(b=-1) == q.QKVP_E_INVALID
    assert call(t=-5) == q.QKVP_E_INVALID
    assert call(out=None) == q.QKVP_E_INVALID
    assert call(out=24) == q.QKVP_E_INVALID                   # output not 16-byte aligned
    assert call(tok=20) == q.QKVP_E_INVALID                   # tok_indptr not 8-byte aligned
    assert call(t=0) == q.QKVP_OK and call(b=0) == q.QKVP_OK  # nothing to do
    g = lib.kv_gather_pages_bf16
    assert g(16, 32, 10, 16, 3, 16, None) == q.QKVP_E_UNSUPPORTED
    assert g(16, 64, 10, 16, -1, 16, None) == q.QKVP_E_INVALID
    assert g(16, 64, 10, 16, 0, 16, None) == q.QKVP_OK
    assert g(None, 64, 10, 16, 3, 16, None) == q.QKVP_E_INVALID
    assert g(16, 64, 10, 16, 3, 8, None) == q.QKVP_E_INVALID


def test_binding_refuses_a_short_or_long_indptr(lib):
    """The C side reads kv_indptr[r + 1] for every request r: the binding checks the length first."""
    lens = np.array([100, 5], np.int32)
    for bad in (np.array([0, 2], np.int32), np.array([0, 2, 3, 4], np.int32)):
        with pytest.raises(ValueError):
            q.mla_decode_plan(bad, lens, 16, q.KV_FP8_E4M3, num_sms=4)
        with pytest.raises(ValueError):
            q.mla_decode_noalloc(bad, lens, 16, q.KV_FP8_E4M3, 16, 16, None, 4, 16, 0.1, 1.0, 16, None,
                                 num_sms=4, stream=0)
    assert plan(np.array([0, 2, 3], np.int32), lens, heads=16, sms=4).status == q.QKVP_OK


def test_plan_of_only_empty_requests(lib):
    """No segments at all: the plan still lists the empty requests (the combine writes their zeros)."""
    p = plan(np.array([0, 1, 1], np.int32), np.array([0, 0], np.int32), heads=16, sms=4)
    assert p.status == q.QKVP_OK and p.num_segments == 0 and p.num_empty_requests == 2
    assert p.total_pages == 0 and p.num_partials == 0


def test_tcgen05_split_charges_request_starts(lib):
    """The tcgen05 plan balances pages plus a fixed cost per request a CTA pair starts (its Q load and
    pipeline refill): pairs that start two requests get fewer pages than pairs that start one, and no
    more requests are cut than under equal page quotas."""
    lens = np.array([32768] * 44, np.int32)
    ptr = np.concatenate([[0], np.cumsum((lens + 63) // 64)]).astype(np.int32)
    tc = plan(ptr, lens, algo=q.ALGO_TCGEN05)
    eq = plan(ptr, lens, algo=q.ALGO_MMA_SYNC)
    assert tc.num_workers == eq.num_workers == 76 and tc.ctas_per_worker == 2
    assert tc.total_pages == eq.total_pages == 44 * 512
    assert tc.num_segments <= eq.num_segments
    mean = -(-tc.total_pages // tc.num_workers)
    assert tc.min_worker_pages < mean <= tc.max_worker_pages          # uneven on purpose
    assert tc.max_worker_pages - tc.min_worker_pages <= 14            # one request start apart
    # a mixed batch: no more request starts than under equal quotas
    rng = np.random.default_rng(0)
    ml = np.exp(rng.uniform(np.log(512), np.log(65536), 64)).astype(np.int32)
    mp = np.concatenate([[0], np.cumsum((ml + 63) // 64)]).astype(np.int32)
    a, b = plan(mp, ml, algo=q.ALGO_TCGEN05), plan(mp, ml, algo=q.ALGO_MMA_SYNC)
    assert a.total_pages == b.total_pages and a.num_segments <= b.num_segments
    # 70 requests of 100 pages over 76 pairs: equal quotas of 93 pages cut 69 requests (two request
    # starts, 93 + 2 x 14 = 121 pages of cost); one whole request per pair costs 100 + 14 = 114, so
    # the budgeted split cuts none and leaves six pairs idle
    sl = np.array([6400] * 70, np.int32)
    sp = np.concatenate([[0], np.cumsum((sl + 63) // 64)]).astype(np.int32)
    a, b = plan(sp, sl, algo=q.ALGO_TCGEN05), plan(sp, sl, algo=q.ALGO_MMA_SYNC)
    assert b.num_segments == 145 and b.max_worker_pages == 93
    assert a.num_segments == 70 and a.max_worker_pages == 100 and a.min_worker_pages == 0


def test_token_major_split_charges_request_starts(lib):
    """The token-major plan (one worker per SM) also balances pages plus a fixed cost of 14 pages per
    request a worker starts: workers are at most one request start apart, and requests that fit a
    worker whole are not cut."""
    lens = np.array([32768] * 44, np.int32)
    ptr = np.concatenate([[0], np.cumsum((lens + 63) // 64)]).astype(np.int32)
    tm = plan(ptr, lens, heads=32, algo=q.ALGO_TCGEN05_TOKENS, sms=152)
    eq = plan(ptr, lens, heads=16, algo=q.ALGO_MMA_SYNC, sms=152)
    assert tm.num_workers == eq.num_workers == 152 and tm.ctas_per_worker == 1
    assert tm.total_pages == eq.total_pages == 44 * 512
    assert tm.num_segments <= eq.num_segments
    assert tm.max_worker_pages - tm.min_worker_pages <= 14
    # 140 requests of 100 pages over 152 workers: equal quotas of 93 pages cut nearly all of them;
    # one whole request per worker costs 100 + 14 = 114 < 93 + 2 x 14, so none is cut
    sl = np.array([6400] * 140, np.int32)
    sp = np.concatenate([[0], np.cumsum((sl + 63) // 64)]).astype(np.int32)
    a = plan(sp, sl, heads=32, algo=q.ALGO_TCGEN05_TOKENS, sms=152)
    b = plan(sp, sl, heads=16, algo=q.ALGO_MMA_SYNC, sms=152)
    assert b.num_segments == 289 and b.max_worker_pages == 93
    assert a.num_segments == 140 and a.max_worker_pages == 100 and a.min_worker_pages == 0


def test_fp8_qk_algo_plans_fp8_pools_only(lib):
    ptr, lens = np.array([0, 2], np.int32), np.array([100], np.int32)
    for kv in (q.KV_FP8_E4M3, q.KV_FP8_PER_TOKEN):
        for heads, per_cta in ((16, 16), (32, 32), (48, 16), (64, 32), (128, 32)):
            p = plan(ptr, lens, heads=heads, kv=kv, algo=q.ALGO_MMA_FP8)
            assert p.status == q.QKVP_OK and p.algo == q.ALGO_MMA_FP8
            assert p.ctas_per_worker == heads // per_cta
    for kv in (q.KV_NVFP4, q.KV_BF16):
        assert plan(ptr, lens, kv=kv, algo=q.ALGO_MMA_FP8).status == q.QKVP_E_UNSUPPORTED
    assert plan(ptr, lens, heads=128).algo == q.ALGO_TCGEN05            # never picked by AUTO


def test_token_major_algo_plans_16_to_64_heads(lib):
    """QKVP_ALGO_TCGEN05_TOKENS: one CTA per SM (workers = SMs, one CTA each), 16-64 heads, quantized
    pools only."""
    ptr, lens = np.array([0, 2], np.int32), np.array([100], np.int32)
    for kv in (q.KV_FP8_E4M3, q.KV_NVFP4, q.KV_FP8_PER_TOKEN):
        for heads in (16, 32, 48, 64):
            p = plan(ptr, lens, heads=heads, kv=kv, algo=q.ALGO_TCGEN05_TOKENS, sms=37)
            assert p.status == q.QKVP_OK and p.algo == q.ALGO_TCGEN05_TOKENS
            assert p.ctas_per_worker == 1 and p.num_workers == 37
        for heads in (80, 128):
            assert plan(ptr, lens, heads=heads, kv=kv, algo=q.ALGO_TCGEN05_TOKENS).status == q.QKVP_E_UNSUPPORTED
    assert plan(ptr, lens, heads=32, kv=q.KV_BF16, algo=q.ALGO_TCGEN05_TOKENS).status == q.QKVP_E_UNSUPPORTED
    assert plan(ptr, lens, heads=16).algo != q.ALGO_TCGEN05_TOKENS
