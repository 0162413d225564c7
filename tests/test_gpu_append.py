"""Quantize-on-append and the device rounding routines against the oracle, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import quantized_kv_paged_gb300 as q
import synth

pytestmark = pytest.mark.gpu


def _special_values():
    v = [0.0, -0.0, 1e-30, -1e-30, 2.0 ** -10, 2.0 ** -9, 3 * 2.0 ** -10, 447.9, 448.0, 449.0, 464.0,
         480.0, 1e6, -1e6, np.inf, -np.inf, np.nan, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 7.0]
    return np.array(v, np.float32)


@pytest.mark.parametrize("fmt", [1, 2])
def test_encode_exhaustive_all_fp32_patterns(qkvp, fmt):
    """Every one of the 2^32 FP32 bit patterns, device rounding vs the oracle's."""
    chunk = 1 << 28
    codes = torch.empty(chunk, dtype=torch.uint8, device="cuda")
    for lo in range(0, 1 << 32, chunk):
        bits = torch.arange(lo, lo + chunk, dtype=torch.int64, device="cuda").to(torch.int32)
        x = bits.view(torch.float32)
        q.qkvp_encode_f32(x, fmt, codes)
        nbad, first = oracle.encode_range_compare(lo, lo + chunk, fmt, codes.cpu().numpy())
        assert nbad == 0, f"fmt {fmt}: {nbad} mismatches, first at bit pattern {first:#010x}"


def _pool(n_slots, width, fill, dev="cuda"):
    return torch.full((n_slots // 64, 64, width), fill, dtype=torch.uint8, device=dev)


@pytest.mark.parametrize("g", [1.0, 0.04464285820722580, 3.0])
@pytest.mark.parametrize("src_kind", ["fp8", "bf16"])
def test_append_nvfp4_bit_exact(qkvp, g, src_kind):
    rng = np.random.default_rng(11)
    n = 4096
    if src_kind == "fp8":
        x = (rng.standard_normal((n, 576)) * np.exp(rng.uniform(-6, 4, (n, 1)))).astype(np.float32)
        x[::7, 5] *= 20
        src = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8)
        src[3, 17] = 0x7F        # NaN byte poisons its block
        src[4, 0:16] = 0         # all-zero block
        src_np, sdt = src.numpy(), oracle.SRC_FP8
    else:
        x = (rng.standard_normal((n, 576)) * np.exp(rng.uniform(-20, 20, (n, 1)))).astype(np.float32)
        sp = _special_values()
        x[0, :sp.size] = sp
        x[1, 16:16 + sp.size] = -sp
        src = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16)
        src_np, sdt = src.numpy().view(np.uint16), oracle.SRC_BF16
    num_pages = 96
    slots = rng.permutation(num_pages * 64)[:n].astype(np.int64)
    slots[10] = -1
    slots[11] = num_pages * 64 + 5            # out of the pool: skipped
    data, scale = _pool(num_pages * 64, 288, 0xAB), _pool(num_pages * 64, 36, 0xCD)
    q.kv_append_quant(src.cuda(), q.SRC_FP8_E4M3 if sdt == 1 else q.SRC_BF16,
                      torch.from_numpy(slots).cuda(), data, scale, q.KV_NVFP4, g)
    torch.cuda.synchronize()
    hd = np.full((num_pages * 64, 288), 0xAB, np.uint8)
    hs = np.full((num_pages * 64, 36), 0xCD, np.uint8)
    ok = slots < num_pages * 64
    oracle.append(src_np[ok], sdt, slots[ok], oracle.KV_NVFP4, g, 64, num_pages, hd, hs)
    gd, gs = data.cpu().numpy().reshape(-1, 288), scale.cpu().numpy().reshape(-1, 36)
    bad = np.nonzero((gd != hd).any(1) | (gs != hs).any(1))[0]
    assert bad.size == 0, f"{bad.size} slots differ, first {bad[:5]}"


@pytest.mark.parametrize("src_kind", ["fp8", "bf16"])
def test_append_fp8_bit_exact(qkvp, src_kind):
    rng = np.random.default_rng(12)
    n = 2048
    x = (rng.standard_normal((n, 576)) * np.exp(rng.uniform(-8, 7, (n, 1)))).astype(np.float32)
    sp = _special_values()
    x[0, :sp.size] = sp
    x[1, :sp.size] = -sp
    if src_kind == "fp8":
        src = torch.from_numpy(np.clip(x, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8)
        src_np, sdt, sd = src.numpy(), oracle.SRC_FP8, q.SRC_FP8_E4M3
    else:
        src = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16)
        src_np, sdt, sd = src.numpy().view(np.uint16), oracle.SRC_BF16, q.SRC_BF16
    num_pages = 40
    slots = rng.permutation(num_pages * 64)[:n].astype(np.int64)
    slots[7] = -3
    pool = _pool(num_pages * 64, 576, 0x5A)
    q.kv_append_quant(src.cuda(), sd, torch.from_numpy(slots).cuda(), pool, None, q.KV_FP8_E4M3, 1.0)
    torch.cuda.synchronize()
    hp = np.full((num_pages * 64, 576), 0x5A, np.uint8)
    oracle.append(src_np, sdt, slots, oracle.KV_FP8, 1.0, 64, num_pages, hp, None)
    assert np.array_equal(pool.cpu().numpy().reshape(-1, 576), hp)


@pytest.mark.parametrize("src_kind", ["fp8", "bf16"])
def test_append_fp8_per_token_bit_exact(qkvp, src_kind):
    rng = np.random.default_rng(13)
    n = 3000
    x = (rng.standard_normal((n, 576)) * np.exp(rng.uniform(-30, 25, (n, 1)))).astype(np.float32)
    x[::5, 100] *= 20
    sp = _special_values()
    if src_kind == "fp8":
        src = torch.from_numpy(np.clip(x, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8)
        src[3, 17] = 0x7F        # NaN byte: the token's scale is NaN, every code 0x7F
        src[4] = 0               # all-zero token: scale 0, codes 0
        src[5, 9] = 0x80         # -0 in an otherwise zero token
        src[5, :9] = 0
        src[5, 10:] = 0
        src[6] = 0x01            # the smallest subnormal everywhere
        src_np, sdt, sd = src.numpy(), oracle.SRC_FP8, q.SRC_FP8_E4M3
    else:
        x[0, :sp.size] = sp      # NaN token
        x[1, :sp.size - 1] = np.delete(sp, np.nonzero(np.isnan(sp))[0][0])   # +-inf: the scale is inf
        x[2] = 0.0
        x[3] = 1e-38
        src = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16)
        src_np, sdt, sd = src.numpy().view(np.uint16), oracle.SRC_BF16, q.SRC_BF16
    num_pages = 60
    slots = rng.permutation(num_pages * 64)[:n].astype(np.int64)
    slots[7] = -3
    slots[8] = num_pages * 64 + 1             # out of the pool: skipped
    pool = torch.full((num_pages, q.PAGE_BYTES_FP8_PER_TOKEN), 0x5A, dtype=torch.uint8, device="cuda")
    q.kv_append_quant(src.cuda(), sd, torch.from_numpy(slots).cuda(), pool, None, q.KV_FP8_PER_TOKEN, 1.0)
    torch.cuda.synchronize()
    hp = np.full((num_pages, oracle.PAGE_BYTES_PT), 0x5A, np.uint8)
    ok = slots < num_pages * 64
    oracle.append(src_np[ok], sdt, slots[ok], oracle.KV_FP8_PT, 1.0, 64, num_pages, hp, None)
    got = pool.cpu().numpy()
    bad = np.nonzero((got != hp).any(1))[0]
    assert bad.size == 0, f"{bad.size} pages differ, first {bad[:5]}"


def test_append_workload_pool_matches_oracle(qkvp):
    """The NVFP4 pool of a decode workload, built through the library and by the oracle."""
    w = synth.build_workload("t", [700, 64, 1], heads=16, pool_pages=20, seed=3, outliers=4, device="cuda")
    from tests.helpers import gpu_pools, oracle_pools
    for g in (1.0, 0.1):
        gd, gs = gpu_pools(w, q.KV_NVFP4, g)
        hd, hs = oracle_pools(w, q.KV_NVFP4, g)
        assert np.array_equal(gd.cpu().numpy(), hd) and np.array_equal(gs.cpu().numpy(), hs)


def test_pool_cast_matches_oracle(qkvp):
    codes = torch.arange(256, dtype=torch.uint8).repeat(64 * 9).cuda()
    out = torch.empty(codes.numel(), dtype=torch.int16, device="cuda")
    q.kv_pool_cast_bf16(codes, out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy().view(np.uint16), oracle.cast_fp8_to_bf16(codes.cpu().numpy()))
