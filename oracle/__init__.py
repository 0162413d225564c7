"""Python access to the FP64 CPU oracle (``qkvp_oracle.cpp``) for paged MLA decode.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package. The product path (``quantized_kv_paged_gb300``) never does, and this
package never imports the product.

``build()`` compiles the oracle with plain g++ (-O2 -ffp-contract=off, no fast-math). Each wrapper
below names the step of the method it states (c1-c6, as written in the C++ source).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qkvp_oracle.cpp")
_OUT = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None
_lock = threading.Lock()

KV_FP8, KV_NVFP4, KV_BF16, KV_FP8_PT = 1, 2, 3, 4
PAGE_BYTES_PT = 64 * (576 + 4)      # c9 page: 64 rows of E4M3 codes, then 64 FP32 token scales
SRC_FP8, SRC_BF16 = 1, 2
D_LATENT, D_V = 576, 512


def build(force: bool = False) -> str:
    """Compile the oracle shared library if it is missing or older than its source."""
    if (not force and os.path.exists(_OUT)
            and os.path.getmtime(_OUT) >= os.path.getmtime(_SRC)):
        return _OUT
    os.makedirs(os.path.dirname(_OUT), exist_ok=True)
    tmp = _OUT + f".{os.getpid()}.tmp"
    cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-pthread", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _OUT)
    return _OUT


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            c = ctypes
            L.qo_e4m3_value.restype = c.c_double
            L.qo_e4m3_value.argtypes = [c.c_uint32]
            L.qo_e2m1_value.restype = c.c_double
            L.qo_e2m1_value.argtypes = [c.c_uint32]
            L.qo_e4m3_encode.restype = c.c_uint8
            L.qo_e4m3_encode.argtypes = [c.c_float]
            L.qo_e2m1_encode.restype = c.c_uint8
            L.qo_e2m1_encode.argtypes = [c.c_float]
            L.qo_encode_array.restype = None
            L.qo_encode_array.argtypes = [c.c_void_p, c.c_int64, c.c_int, c.c_void_p, c.c_int]
            L.qo_encode_range_compare.restype = c.c_int64
            L.qo_encode_range_compare.argtypes = [c.c_uint64, c.c_uint64, c.c_int, c.c_void_p,
                                                  c.POINTER(c.c_uint64), c.c_int]
            L.qo_nvfp4_block.restype = None
            L.qo_nvfp4_block.argtypes = [c.c_void_p, c.c_float, c.c_void_p, c.c_void_p]
            L.qo_quant_tokens.restype = c.c_int
            L.qo_quant_tokens.argtypes = [c.c_void_p, c.c_int, c.c_int64, c.c_int, c.c_float,
                                          c.c_void_p, c.c_void_p, c.c_int]
            L.qo_append.restype = c.c_int
            L.qo_append.argtypes = [c.c_void_p, c.c_int, c.c_int64, c.c_void_p, c.c_int, c.c_float,
                                    c.c_int, c.c_int64, c.c_void_p, c.c_void_p]
            L.qo_dequant_slot.restype = None
            L.qo_dequant_slot.argtypes = [c.c_void_p, c.c_void_p, c.c_int, c.c_double, c.c_int64,
                                          c.c_void_p]
            L.qo_mla_decode.restype = c.c_int
            L.qo_mla_decode.argtypes = [c.c_void_p, c.c_int, c.c_int, c.c_void_p, c.c_void_p,
                                        c.c_int, c.c_int, c.c_int64, c.c_void_p, c.c_void_p,
                                        c.c_void_p, c.c_double, c.c_double, c.c_void_p, c.c_int64,
                                        c.c_void_p, c.c_void_p, c.c_int]
            L.qo_lse_merge.restype = None
            L.qo_lse_merge.argtypes = [c.c_int, c.c_int, c.c_void_p, c.c_void_p, c.c_void_p,
                                       c.c_void_p]
            L.qo_cast_fp8_to_bf16.restype = None
            L.qo_cast_fp8_to_bf16.argtypes = [c.c_void_p, c.c_int64, c.c_void_p]
            L.qo_gather_fp8.argtypes = [c.c_void_p, c.c_void_p, c.c_int, c.c_float, c.c_int, c.c_int64,
                                        c.c_void_p, c.c_void_p, c.c_int64, c.c_void_p, c.c_int, c.c_void_p]
            L.qo_gather_fp8.restype = c.c_int64
            L.qo_gather_pages_bf16.argtypes = [c.c_void_p, c.c_int, c.c_int64, c.c_void_p, c.c_int64,
                                               c.c_void_p]
            L.qo_hardware_threads.restype = c.c_int
            _lib = L
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def threads() -> int:
    return max(1, int(lib().qo_hardware_threads()))


# ---- c1 / c2 / c3 codecs -------------------------------------------------------------------------

def e4m3_value(code: int) -> float:
    return lib().qo_e4m3_value(code)


def e2m1_value(code: int) -> float:
    return lib().qo_e2m1_value(code)


def e4m3_encode(x: float) -> int:
    return int(lib().qo_e4m3_encode(x))


def e2m1_encode(x: float) -> int:
    return int(lib().qo_e2m1_encode(x))


def encode_array(x: np.ndarray, fmt: int) -> np.ndarray:
    """fmt 1: E4M3 (c2); fmt 2: E2M1 (c3 step 5). One code byte per FP32 input."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().qo_encode_array(_p(x), x.size, fmt, _p(out), threads())
    return out


def encode_range_compare(lo: int, hi: int, fmt: int, codes: np.ndarray):
    """Compare `codes` against the oracle's encoding of every FP32 bit pattern in [lo, hi)."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    assert codes.size == hi - lo
    first = ctypes.c_uint64(0)
    nbad = lib().qo_encode_range_compare(lo, hi, fmt, _p(codes), ctypes.byref(first), threads())
    return int(nbad), int(first.value)


def nvfp4_block(x16, g: float):
    """c3 on one block: returns (8 packed bytes, 1 scale byte)."""
    x = np.ascontiguousarray(x16, dtype=np.float32)
    assert x.size == 16
    packed = np.zeros(8, dtype=np.uint8)
    scale = np.zeros(1, dtype=np.uint8)
    lib().qo_nvfp4_block(_p(x), g, _p(packed), _p(scale))
    return packed, int(scale[0])


def quant_tokens(src: np.ndarray, src_dtype: int, kv_dtype: int, g: float = 1.0):
    """Token-major quantisation. src: uint8 [n,576] (FP8) or uint16 [n,576] (BF16 bits).

    Returns data [n,576] (FP8), (data [n,288], scales [n,36]) (NVFP4) or (codes [n,576], token
    scales float32 [n]) (FP8_PT, c9)."""
    src = np.ascontiguousarray(src)
    n = src.shape[0]
    if kv_dtype == KV_FP8:
        data = np.empty((n, D_LATENT), dtype=np.uint8)
        scale = np.empty((1,), dtype=np.uint8)
    elif kv_dtype == KV_FP8_PT:
        data = np.empty((n, D_LATENT), dtype=np.uint8)
        scale = np.empty((n,), dtype=np.float32)
    else:
        data = np.empty((n, D_LATENT // 2), dtype=np.uint8)
        scale = np.empty((n, D_LATENT // 16), dtype=np.uint8)
    rc = lib().qo_quant_tokens(_p(src), src_dtype, n, kv_dtype, g, _p(data), _p(scale), threads())
    if rc:
        raise ValueError(f"qo_quant_tokens rc={rc}")
    return data if kv_dtype == KV_FP8 else (data, scale)


def pt_pool(num_pages: int) -> np.ndarray:
    """An empty (all-zero) per-token-scaled FP8 pool of `num_pages` c9 pages."""
    return np.zeros((num_pages, PAGE_BYTES_PT), dtype=np.uint8)


def append(src: np.ndarray, src_dtype: int, slots: np.ndarray, kv_dtype: int, g: float,
           page_size: int, num_pages: int, pool_data: np.ndarray, pool_scale: np.ndarray | None):
    """Quantize-on-append into host pools (modified in place)."""
    src = np.ascontiguousarray(src)
    slots = np.ascontiguousarray(slots, dtype=np.int64)
    ps = _p(pool_scale) if pool_scale is not None else None
    rc = lib().qo_append(_p(src), src_dtype, src.shape[0], _p(slots), kv_dtype, g, page_size,
                         num_pages, _p(pool_data), ps)
    if rc:
        raise ValueError(f"qo_append rc={rc}")


def dequant_slot(kv_data: np.ndarray, kv_scale, kv_dtype: int, g: float, slot: int) -> np.ndarray:
    x = np.empty(D_LATENT, dtype=np.float64)
    ps = _p(kv_scale) if kv_scale is not None else None
    lib().qo_dequant_slot(_p(kv_data), ps, kv_dtype, g, slot, _p(x))
    return x


def mla_decode(q_bf16_bits: np.ndarray, kv_data: np.ndarray, kv_scale, kv_dtype: int,
               page_size: int, num_pages: int, kv_indptr, kv_indices, kv_len, sm_scale: float,
               g: float = 1.0, pairs=None, nthreads: int | None = None):
    """c5: FP64 decode attention. q: uint16 BF16 bits [B,H,576]. pairs: optional int32 [n,2] of
    (request, head); default all. Returns (o [n,512] float64, lse [n] float64)."""
    q = np.ascontiguousarray(q_bf16_bits, dtype=np.uint16)
    B, H = q.shape[0], q.shape[1]
    kv_indptr = np.ascontiguousarray(kv_indptr, dtype=np.int32)
    kv_indices = np.ascontiguousarray(kv_indices, dtype=np.int32)
    kv_len = np.ascontiguousarray(kv_len, dtype=np.int32)
    if pairs is None:
        n = B * H
        pp = None
    else:
        pairs = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
        n = pairs.shape[0]
        pp = _p(pairs)
    o = np.empty((n, D_V), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    ps = _p(kv_scale) if kv_scale is not None else None
    rc = lib().qo_mla_decode(_p(q), B, H, _p(np.ascontiguousarray(kv_data)), ps, kv_dtype,
                             page_size, num_pages, _p(kv_indptr), _p(kv_indices), _p(kv_len),
                             float(np.float32(sm_scale)), float(np.float32(g)), pp, n, _p(o),
                             _p(lse), nthreads or threads())
    if rc:
        raise ValueError(f"qo_mla_decode rc={rc}")
    return o, lse


def lse_merge(o_parts: np.ndarray, lse_parts: np.ndarray):
    """c6: merge normalised partial outputs by their log-sum-exp."""
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    n, dv = o_parts.shape
    o = np.empty(dv, dtype=np.float64)
    lse = np.empty(1, dtype=np.float64)
    lib().qo_lse_merge(n, dv, _p(o_parts), _p(lse_parts), _p(o), _p(lse))
    return o, float(lse[0])


def cast_fp8_to_bf16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.uint8)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().qo_cast_fp8_to_bf16(_p(x), x.size, _p(out))
    return out


def gather_fp8(kv_data: np.ndarray, kv_scale, kv_dtype: int, g: float, page_size: int, num_pages: int,
               kv_indptr, kv_indices, tok_indptr):
    """c7: gather each request's tokens into a contiguous E4M3 workspace [tok_indptr[-1], 576]
    (FP8 copied, NVFP4 dequantized and re-encoded). Returns (workspace, rows from bad page ids)."""
    kv_indptr = np.ascontiguousarray(kv_indptr, dtype=np.int32)
    kv_indices = np.ascontiguousarray(kv_indices, dtype=np.int32)
    tok_indptr = np.ascontiguousarray(tok_indptr, dtype=np.int64)
    out = np.empty((int(tok_indptr[-1]), D_LATENT), dtype=np.uint8)
    ps = _p(np.ascontiguousarray(kv_scale)) if kv_scale is not None else None
    bad = lib().qo_gather_fp8(_p(np.ascontiguousarray(kv_data)), ps, kv_dtype, float(np.float32(g)), page_size,
                              num_pages, _p(kv_indptr), _p(kv_indices), kv_indices.size, _p(tok_indptr),
                              len(tok_indptr) - 1, _p(out))
    return out, int(bad)


def gather_pages_bf16(pool: np.ndarray, page_ids, page_size: int = 64) -> np.ndarray:
    """c8: pages page_ids of an FP8 pool [P, page_size, 576], cast to BF16 bits [n, page_size, 576]."""
    pool = np.ascontiguousarray(pool, dtype=np.uint8)
    ids = np.ascontiguousarray(page_ids, dtype=np.int32)
    out = np.empty((ids.size, page_size, D_LATENT), dtype=np.uint16)
    lib().qo_gather_pages_bf16(_p(pool), page_size, pool.shape[0], _p(ids), ids.size, _p(out))
    return out
