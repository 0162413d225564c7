"""Python binding of libqkvp: paged MLA decode over a quantized (FP8 E4M3 / NVFP4) latent KV cache.

Argument marshalling only: every function below forwards to the C entry point of the same name
(``include/qkvp.h``) with raw device pointers and the current torch CUDA stream. All computation runs
in the library's CUDA kernels. There is no fallback: if the library is missing, ``load()`` raises.
PyTorch is used for device memory and streams.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libqkvp.so")

QKVP_OK, QKVP_E_INVALID, QKVP_E_UNSUPPORTED, QKVP_E_WORKSPACE, QKVP_E_CUDA = 0, -1, -2, -3, -4
KV_FP8_E4M3, KV_NVFP4, KV_BF16, KV_FP8_PER_TOKEN = 1, 2, 3, 4
PAGE_BYTES_FP8_PER_TOKEN = 64 * (576 + 4)   # 64 rows of E4M3 codes, then 64 FP32 token scales
SRC_FP8_E4M3, SRC_BF16 = 1, 2
ALGO_AUTO, ALGO_MMA_SYNC, ALGO_TCGEN05, ALGO_MMA_FP8, ALGO_TCGEN05_TOKENS = 0, 1, 2, 3, 4
LATENT_DIM, V_DIM, PAGE_SIZE = 576, 512, 64

EXPORTS = ["kv_append_quant", "mla_decode_plan", "mla_decode_run", "mla_decode_attend",
           "mla_decode_combine", "mla_decode_noalloc", "kv_pool_cast_bf16", "kv_gather_fp8",
           "kv_gather_pages_bf16", "qkvp_encode_f32", "qkvp_status_string", "qkvp_version"]


class qkvp_plan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "num_heads", "page_size", "kv_dtype", "algo", "num_workers", "ctas_per_worker",
        "num_segments", "num_split_requests", "num_empty_requests", "max_worker_pages",
        "min_worker_pages", "num_partials", "max_request_segments",
        "num_wide_requests")] + [
        ("total_pages", ctypes.c_int64), ("total_tokens", ctypes.c_int64),
        ("workspace_bytes", ctypes.c_uint64), ("table_bytes", ctypes.c_uint64),
        ("partial_o_offset", ctypes.c_uint64), ("partial_lse_offset", ctypes.c_uint64),
        ("status_offset", ctypes.c_uint64), ("magic", ctypes.c_uint64)]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class QkvpError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")
        self.status = status


_lib = None
_lock = threading.Lock()


def load(path: str | None = None):
    """Load libqkvp.so (built by ``quantized_kv_paged_gb300.build``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"libqkvp.so not found at {p}: run quantized_kv_paged_gb300.build.build()")
        L = ctypes.CDLL(p)
        c = ctypes
        vp, i32, i64, u64, f32 = c.c_void_p, c.c_int32, c.c_int64, c.c_uint64, c.c_float
        L.kv_append_quant.argtypes = [vp, i32, i64, vp, vp, vp, i32, f32, i32, i64, vp]
        L.mla_decode_plan.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, u64, vp,
                                      c.POINTER(qkvp_plan)]
        L.mla_decode_run.argtypes = [c.POINTER(qkvp_plan), vp, vp, vp, i64, vp, f32, f32, vp, vp,
                                     vp, u64, vp]
        L.mla_decode_attend.argtypes = L.mla_decode_run.argtypes
        L.mla_decode_combine.argtypes = [c.POINTER(qkvp_plan), f32, vp, vp, vp, u64, vp]
        L.mla_decode_noalloc.argtypes = [vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, i64, vp, f32,
                                         f32, vp, vp, vp]
        L.kv_pool_cast_bf16.argtypes = [vp, i64, vp, vp]
        L.kv_gather_fp8.argtypes = [vp, vp, i32, f32, i32, i64, vp, vp, i64, vp, i32, i64, vp, vp]
        L.kv_gather_pages_bf16.argtypes = [vp, i32, i64, vp, i64, vp, vp]
        L.qkvp_encode_f32.argtypes = [vp, i64, i32, vp, vp]
        L.qkvp_status_string.restype = c.c_char_p
        L.qkvp_status_string.argtypes = [c.c_int]
        for fn in ("kv_append_quant", "mla_decode_plan", "mla_decode_run", "mla_decode_attend",
                   "mla_decode_combine", "mla_decode_noalloc", "kv_pool_cast_bf16", "kv_gather_fp8",
                   "kv_gather_pages_bf16", "qkvp_encode_f32", "qkvp_version"):
            getattr(L, fn).restype = c.c_int
        _lib = L
        return L


def status_string(status: int) -> str:
    return load().qkvp_status_string(status).decode()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream(stream):
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    return torch.cuda.current_stream().cuda_stream


def _table(kv_indptr, kv_len):
    """The host page table as contiguous int32 arrays; kv_indptr must have len(kv_len) + 1 entries
    (the library reads kv_indptr[r + 1] for every request r)."""
    indptr = np.ascontiguousarray(kv_indptr, dtype=np.int32)
    lens = np.ascontiguousarray(kv_len, dtype=np.int32)
    if indptr.ndim != 1 or lens.ndim != 1 or indptr.shape[0] != lens.shape[0] + 1:
        raise ValueError(f"kv_indptr needs len(kv_len) + 1 = {lens.shape[0] + 1} entries, got {indptr.shape}")
    return indptr, lens


def _check(fn, status, raise_on_error):
    if status != QKVP_OK and raise_on_error:
        raise QkvpError(fn, status)
    return status


def kv_append_quant(src, src_dtype: int, slot_mapping, kv_data, kv_scale, kv_dtype: int,
                    global_scale: float = 1.0, num_pages: int | None = None,
                    page_size: int = PAGE_SIZE, stream=None, raise_on_error: bool = True) -> int:
    """Quantize-on-append of src [n, 576] into the paged pool at slot_mapping (see qkvp.h)."""
    n = int(src.shape[0]) if src is not None else 0
    if num_pages is None:
        num_pages = int(kv_data.shape[0])
    st = load().kv_append_quant(_ptr(src), src_dtype, n, _ptr(slot_mapping), _ptr(kv_data),
                                _ptr(kv_scale), kv_dtype, float(global_scale), page_size,
                                int(num_pages), _stream(stream))
    return _check("kv_append_quant", st, raise_on_error)


def mla_decode_plan(kv_indptr, kv_len, num_heads: int, kv_dtype: int, num_sms: int = 0,
                    min_splits: int = 0, algo: int = ALGO_AUTO, workspace=None,
                    page_size: int = PAGE_SIZE, stream=None, raise_on_error: bool = True):
    """Plan the split; with workspace=None only sizes are computed. Returns a qkvp_plan."""
    indptr, lens = _table(kv_indptr, kv_len)
    plan = qkvp_plan()
    ws = _ptr(workspace)
    nbytes = int(workspace.numel() * workspace.element_size()) if workspace is not None else 0
    st = load().mla_decode_plan(indptr.ctypes.data, lens.ctypes.data, int(lens.shape[0]),
                                num_heads, page_size, kv_dtype, num_sms, min_splits, algo, ws,
                                nbytes, _stream(stream) if ws else None, ctypes.byref(plan))
    _check("mla_decode_plan", st, raise_on_error)
    plan.status = st
    return plan


def mla_decode_run(plan: qkvp_plan, q, kv_data, kv_scale, num_pages: int, kv_indices,
                   sm_scale: float, global_scale: float, out, lse, workspace, stream=None,
                   raise_on_error: bool = True) -> int:
    """Decode one layer: out [B, H, 512] bf16 and lse [B, H] float32 (lse may be None)."""
    nbytes = int(workspace.numel() * workspace.element_size()) if workspace is not None else 0
    st = load().mla_decode_run(ctypes.byref(plan), _ptr(q), _ptr(kv_data), _ptr(kv_scale),
                               int(num_pages), _ptr(kv_indices), float(sm_scale),
                               float(global_scale), _ptr(out), _ptr(lse), _ptr(workspace), nbytes,
                               _stream(stream))
    return _check("mla_decode_run", st, raise_on_error)


def mla_decode_attend(plan: qkvp_plan, q, kv_data, kv_scale, num_pages: int, kv_indices,
                      sm_scale: float, global_scale: float, out, lse, workspace, stream=None,
                      raise_on_error: bool = True) -> int:
    """The split-KV decode kernel alone (first half of mla_decode_run)."""
    nbytes = int(workspace.numel() * workspace.element_size())
    st = load().mla_decode_attend(ctypes.byref(plan), _ptr(q), _ptr(kv_data), _ptr(kv_scale),
                                  int(num_pages), _ptr(kv_indices), float(sm_scale),
                                  float(global_scale), _ptr(out), _ptr(lse), _ptr(workspace),
                                  nbytes, _stream(stream))
    return _check("mla_decode_attend", st, raise_on_error)


def mla_decode_combine(plan: qkvp_plan, global_scale: float, out, lse, workspace, stream=None,
                       raise_on_error: bool = True) -> int:
    """The log-sum-exp merge of split partials (second half of mla_decode_run)."""
    nbytes = int(workspace.numel() * workspace.element_size())
    st = load().mla_decode_combine(ctypes.byref(plan), float(global_scale), _ptr(out), _ptr(lse),
                                   _ptr(workspace), nbytes, _stream(stream))
    return _check("mla_decode_combine", st, raise_on_error)


def mla_decode_noalloc(kv_indptr, kv_len, num_heads: int, kv_dtype: int, q, kv_data, kv_scale,
                       num_pages: int, kv_indices, sm_scale: float, global_scale: float, out, lse,
                       num_sms: int = 0, min_splits: int = 0, stream=None,
                       raise_on_error: bool = True) -> int:
    """Plan + decode with the library's fixed scratch array, for callers that cannot allocate
    device memory (see qkvp.h for the size limit and the sharing rules)."""
    indptr, lens = _table(kv_indptr, kv_len)
    st = load().mla_decode_noalloc(indptr.ctypes.data, lens.ctypes.data, int(lens.shape[0]), num_heads,
                                   kv_dtype, num_sms, min_splits, _ptr(q), _ptr(kv_data),
                                   _ptr(kv_scale), int(num_pages), _ptr(kv_indices), float(sm_scale),
                                   float(global_scale), _ptr(out), _ptr(lse), _stream(stream))
    return _check("mla_decode_noalloc", st, raise_on_error)


def kv_pool_cast_bf16(src, out, stream=None, raise_on_error: bool = True) -> int:
    """The cast-then-attend baseline's pool-wide FP8 -> BF16 cast."""
    st = load().kv_pool_cast_bf16(_ptr(src), int(src.numel()), _ptr(out), _stream(stream))
    return _check("kv_pool_cast_bf16", st, raise_on_error)


def kv_gather_fp8(kv_data, kv_scale, kv_dtype: int, global_scale: float, kv_indptr, kv_indices, tok_indptr,
                  out, num_pages: int | None = None, page_size: int = PAGE_SIZE, stream=None,
                  raise_on_error: bool = True) -> int:
    """Extend-path gather of each request's tokens into the FP8 workspace out [T, 576] (see qkvp.h).
    kv_indptr / kv_indices int32 and tok_indptr int64 are device tensors."""
    if num_pages is None:
        num_pages = int(kv_data.shape[0])
    batch = int(tok_indptr.shape[0]) - 1
    st = load().kv_gather_fp8(_ptr(kv_data), _ptr(kv_scale), kv_dtype, float(global_scale), page_size,
                              int(num_pages), _ptr(kv_indptr), _ptr(kv_indices), int(kv_indices.numel()),
                              _ptr(tok_indptr), batch, int(out.shape[0]), _ptr(out), _stream(stream))
    return _check("kv_gather_fp8", st, raise_on_error)


def kv_gather_pages_bf16(kv_data, page_ids, out, num_pages: int | None = None, page_size: int = PAGE_SIZE,
                         stream=None, raise_on_error: bool = True) -> int:
    """Gather-then-cast baseline: pool pages page_ids (device int32) cast into out [n, 64, 576] BF16."""
    if num_pages is None:
        num_pages = int(kv_data.shape[0])
    st = load().kv_gather_pages_bf16(_ptr(kv_data), page_size, int(num_pages), _ptr(page_ids),
                                     int(page_ids.numel()), _ptr(out), _stream(stream))
    return _check("kv_gather_pages_bf16", st, raise_on_error)


def qkvp_encode_f32(x, fmt: int, codes, stream=None, raise_on_error: bool = True) -> int:
    """Device E4M3 (fmt 1) / E2M1 (fmt 2) rounding of FP32 values, one code byte each."""
    st = load().qkvp_encode_f32(_ptr(x), int(x.numel()), fmt, _ptr(codes), _stream(stream))
    return _check("qkvp_encode_f32", st, raise_on_error)


def qkvp_version() -> int:
    return load().qkvp_version()
