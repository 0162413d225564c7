"""Why the decode kernels multiply in FP16, not FP8 (the FP8-compute variant the pages mention as an
option of the decode path: "SGLang x Qwen x NVIDIA ... NVFP4 KV Cache", section "SGLang
implementation", item 3, dequantize on the fly to FP8 or BF16; the extend path of item 2 attends in
FP8).

On a request of the benchmark's shape (32K tokens, N(0, 1) latents with four x20 outlier channels,
N(0, 1) BF16 queries), attention is evaluated with the operands the tensor cores would see and exact
products summed in FP64; the FP64 oracle is the reference. The E4M3 roundings are the oracle's
encoder. Outcomes, against the stated bound (max-abs 2e-2 over half a BF16 ulp):
  - Q rounded to E4M3 (per-head power-of-two scale): the outlier channels of K amplify the rounding of
    q, the excess is two orders of magnitude over the bound;
  - P rounded to E4M3 (P x 2^8, FP16-exact everything else): over the bound;
  - Q as a two-term E4M3 sum (q = hi + lo / 16) with FP16 P: within the bound. That split doubles the
    Q.K^T MMAs, which is the FP16 MMA count again: FP8 operands cannot raise the tensor ceiling of
    this decode within the tolerance.
The two-term form is the library's FP8 Q.K^T variant (QKVP_ALGO_MMA_FP8); its GPU parity tests are in
test_gpu_decode.py.
"""
import numpy as np
import pytest

import oracle
import synth

MAX_ABS = 2e-2
_E4M3 = np.array([oracle.e4m3_value(c) for c in range(256)])


def _e4m3(x: np.ndarray) -> np.ndarray:
    codes = oracle.encode_array(np.ascontiguousarray(x, dtype=np.float64).ravel(), 1)   # fmt 1: E4M3
    return _E4M3[codes].reshape(x.shape)


def _f16(x: np.ndarray) -> np.ndarray:
    return x.astype(np.float16).astype(np.float64)


def _bf16_excess(o: np.ndarray, ref: np.ndarray) -> float:
    ob = o.astype(np.float32)
    ob = (ob.view(np.uint32) + 0x7FFF + ((ob.view(np.uint32) >> 16) & 1)) & 0xFFFF0000   # RNE to BF16
    ob = ob.astype(np.uint32).view(np.float32).astype(np.float64)
    a = np.abs(ref)
    half_ulp = 0.5 * 2.0 ** (np.floor(np.log2(np.maximum(a, 2.0 ** -126))) - 7)
    return float(np.maximum(np.abs(ob - ref) - half_ulp, 0.0).max())


@pytest.fixture(scope="module")
def case():
    lens = [32768]
    w = synth.build_workload("fp8prec", lens, heads=16, pool_pages=520, seed=3, outliers=4, device="cpu")
    pool = w.pool_fp8.numpy()
    q_bits = w.q.view(__import__("torch").int16).numpy().view(np.uint16)
    o_ref, _ = oracle.mla_decode(q_bits, pool, None, oracle.KV_FP8, 64, w.num_pages, w.kv_indptr,
                                 w.kv_indices, w.kv_len, w.sm_scale, 1.0, None)
    kv = _E4M3[pool.reshape(w.num_pages, 64, 576)[w.kv_indices[: 32768 // 64]].reshape(-1, 576)]
    q = (q_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64).reshape(16, 576)
    return q, kv, w.sm_scale, o_ref.reshape(16, 512)


def _attend(q, kv, sm_scale, p_round):
    s = (q @ kv.T) * sm_scale
    p = np.exp(s - s.max(1, keepdims=True))
    p = p_round(p)
    return (p @ kv[:, :512]) / p.sum(1, keepdims=True)


def _q_scale(q):
    return 2.0 ** np.floor(np.log2(448.0 / np.abs(q).max(1, keepdims=True)))


def test_reference_arithmetic_meets_the_bound(case):
    q, kv, sm, ref = case
    assert _bf16_excess(_attend(_f16(q * _q_scale(q)) / _q_scale(q), kv, sm, _f16), ref) < 1e-3


def test_fp8_query_breaks_the_bound(case):
    q, kv, sm, ref = case
    sc = _q_scale(q)
    assert _bf16_excess(_attend(_e4m3(q * sc) / sc, kv, sm, _f16), ref) > 10 * MAX_ABS


def test_fp8_probabilities_break_the_bound(case):
    q, kv, sm, ref = case
    sc = _q_scale(q)
    assert _bf16_excess(_attend(_f16(q * sc) / sc, kv, sm, lambda p: _e4m3(p * 256.0) / 256.0), ref) > MAX_ABS


def test_two_term_fp8_query_meets_the_bound(case):
    q, kv, sm, ref = case
    sc = _q_scale(q)
    hi = _e4m3(q * sc)
    lo = _e4m3((q * sc - hi) * 16.0) / 16.0
    assert _bf16_excess(_attend((hi + lo) / sc, kv, sm, _f16), ref) < MAX_ABS
