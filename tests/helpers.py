"""Helpers shared by the GPU parity tests: build device and oracle pools for a workload, run the
CUDA path through the C ABI, run the oracle, and compare under the stated tolerance."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import quantized_kv_paged_gb300 as q
import synth

KV_NAMES = {q.KV_FP8_E4M3: "fp8", q.KV_NVFP4: "nvfp4", q.KV_BF16: "bf16", q.KV_FP8_PER_TOKEN: "fp8_per_token"}

# Tolerance on BF16 outputs, from the stated target: max-abs 2e-2, mean-abs 2e-3. It is applied to
# the excess of |out - o_ref| over half a BF16 ulp of o_ref (the rounding any BF16 output carries);
# workloads without outlier channels (|o| < 2) are also held to it on the raw difference.
MAX_ABS, MEAN_ABS = 2e-2, 2e-3
LSE_ATOL, LSE_RTOL = 2e-3, 1e-4


def gpu_pools(w: synth.Workload, kv: int, g: float = 1.0):
    """(kv_data, kv_scale) on the GPU for kv dtype `kv`, built through the library."""
    dev = w.pool_fp8.device
    if kv == q.KV_FP8_E4M3:
        return w.pool_fp8, None
    if kv == q.KV_NVFP4:
        data = torch.full((w.num_pages, 64, 288), 0xFF, dtype=torch.uint8, device=dev)
        scale = torch.full((w.num_pages, 64, 36), 0x7F, dtype=torch.uint8, device=dev)
        q.kv_append_quant(w.src_fp8, q.SRC_FP8_E4M3, w.slots, data, scale, q.KV_NVFP4, g)
        return data, scale
    if kv == q.KV_FP8_PER_TOKEN:
        # slots never appended hold NaN codes and NaN scales: decode must never read them
        data = torch.full((w.num_pages, q.PAGE_BYTES_FP8_PER_TOKEN), 0xFF, dtype=torch.uint8, device=dev)
        q.kv_append_quant(w.src_fp8, q.SRC_FP8_E4M3, w.slots, data, None, q.KV_FP8_PER_TOKEN, 1.0)
        return data, None
    out = torch.empty((w.num_pages, 64, 576), dtype=torch.int16, device=dev)
    q.kv_pool_cast_bf16(w.pool_fp8, out)
    return out, None


def oracle_pools(w: synth.Workload, kv: int, g: float = 1.0):
    """The same pools built on the host by the oracle from the generated FP8 bytes."""
    pool = w.pool_fp8.cpu().numpy()
    if kv == q.KV_FP8_E4M3:
        return pool, None
    if kv == q.KV_NVFP4:
        data = np.full((w.num_pages * 64, 288), 0xFF, np.uint8)
        scale = np.full((w.num_pages * 64, 36), 0x7F, np.uint8)
        d, s = oracle.quant_tokens(w.src_fp8.cpu().numpy(), oracle.SRC_FP8, oracle.KV_NVFP4, g)
        slots = w.slots.cpu().numpy()
        data[slots] = d
        scale[slots] = s
        return data.reshape(w.num_pages, 64, 288), scale.reshape(w.num_pages, 64, 36)
    if kv == q.KV_FP8_PER_TOKEN:
        # the oracle's quantisation (threaded), placed at the slots by the c9 page layout
        data = np.full((w.num_pages, oracle.PAGE_BYTES_PT), 0xFF, np.uint8)
        codes, sig = oracle.quant_tokens(w.src_fp8.cpu().numpy(), oracle.SRC_FP8, oracle.KV_FP8_PT)
        slots = w.slots.cpu().numpy()
        page, off = slots // 64, slots % 64
        data[:, :64 * 576].reshape(w.num_pages, 64, 576)[page, off] = codes
        data[:, 64 * 576:].view(np.float32).reshape(w.num_pages, 64)[page, off] = sig
        return data, None
    return oracle.cast_fp8_to_bf16(pool), None


def gpu_decode(w: synth.Workload, kv: int, pools, g: float = 1.0, num_sms: int = 0,
               min_splits: int = 0, algo: int = 0, lens=None, indices=None):
    dev = w.pool_fp8.device
    lens = w.kv_len if lens is None else lens
    plan = q.mla_decode_plan(w.kv_indptr, lens, w.heads, kv, num_sms=num_sms,
                             min_splits=min_splits, algo=algo)
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=dev)
    plan = q.mla_decode_plan(w.kv_indptr, lens, w.heads, kv, num_sms=num_sms,
                             min_splits=min_splits, algo=algo, workspace=ws)
    out = torch.full((w.batch, w.heads, 512), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((w.batch, w.heads), float("nan"), dtype=torch.float32, device=dev)
    idx = torch.from_numpy(w.kv_indices if indices is None else indices).to(dev)
    q.mla_decode_run(plan, w.q, pools[0], pools[1], w.num_pages, idx, w.sm_scale, g, out, lse, ws)
    torch.cuda.synchronize()
    status = int(ws[plan.status_offset:plan.status_offset + 4].view(torch.int32).item())
    assert status == 0, f"decode kernel gave up waiting (status {status:#x})"
    return out, lse, plan


def oracle_decode(w: synth.Workload, kv: int, host_pools, g: float = 1.0, pairs=None, lens=None):
    qb = w.q.cpu().view(torch.int16).numpy().view(np.uint16)
    return oracle.mla_decode(qb, host_pools[0], host_pools[1], kv, 64, w.num_pages, w.kv_indptr,
                             w.kv_indices, w.kv_len if lens is None else lens, w.sm_scale, g, pairs)


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    a = np.abs(x)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 0.5 * 2.0 ** (e - 7)


def compare(out: np.ndarray, lse: np.ndarray, o_ref: np.ndarray, lse_ref: np.ndarray, raw: bool = False):
    """Returns a dict of error statistics and asserts the tolerance."""
    out = out.astype(np.float64)
    assert np.all(np.isfinite(out)), "non-finite output"
    err = np.abs(out - o_ref)
    excess = np.maximum(0.0, err - half_ulp_bf16(o_ref))
    floor = np.abs(torch.from_numpy(o_ref).to(torch.bfloat16).to(torch.float64).numpy() - o_ref)
    stats = {"raw_max": float(err.max()), "raw_mean": float(err.mean()),
             "excess_max": float(excess.max()), "excess_mean": float(excess.mean()),
             "floor_max": float(floor.max()), "o_absmax": float(np.abs(o_ref).max())}
    e = err if raw else excess
    assert e.max() <= MAX_ABS, stats
    assert e.mean() <= MEAN_ABS, stats
    fin = np.isfinite(lse_ref)
    assert np.array_equal(fin, np.isfinite(lse)), "lse finiteness differs"
    if fin.any():
        d = np.abs(lse[fin] - lse_ref[fin])
        assert np.all(d <= LSE_ATOL + LSE_RTOL * np.abs(lse_ref[fin])), float(d.max())
    if (~fin).any():
        assert np.all(lse[~fin] == lse_ref[~fin])
    return stats
