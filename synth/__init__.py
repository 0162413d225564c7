"""Seeded synthetic workloads for paged MLA decode over a quantized latent KV cache.

This module is shared by the tests, the benchmark and the oracle checks. It draws random numbers and
lays bytes out in pages. It holds none of the method's arithmetic: no block quantisation, no
dequantisation, no attention. The one number-format step it takes is rounding the Gaussian latent
to FP8 E4M3 with torch's own ``float8_e4m3fn`` cast. That stands in for the model whose KV cache is
FP8 ("the KV cache is kept as float8_e4m3fn", The FP8 KV Cache Wall, section "Context and
Motivation").

Random numbers come from SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014; finaliser constants as published by Vigna). It is used as a counter-based
generator: value i of stream s is the finaliser applied to key(seed, s) + (i + 1) * golden. Normals
come from Box-Muller on pairs of 53-bit uniforms. The same counter gives the same number on any
device, up to the last ulp of torch's log/cos/sin on that device. The oracle therefore always reads
the exact bytes that were generated (copied to the host), never a regenerated copy.

Shapes follow the pages' problem statement: each token stores one 576-wide latent, 512 "nope" dims
(kv_lora_rank) and 64 rope dims (The Smoking Gun, section "The Investigation Leading to This
Message": shape [495552, 1, 576] with 576 = 512 + 64). Pages hold 64 tokens.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

D_LATENT = 576          # kv_lora_rank 512 + qk_rope_head_dim 64
D_V = 512               # V is the first 512 latent dims
PAGE = 64               # tokens per page
FP8_NAN = 0x7F          # E4M3FN NaN byte, used to poison slots that no request owns

_M64 = (1 << 64) - 1


def _i64(x: int) -> int:
    """Python int -> the int64 with the same low 64 bits."""
    x &= _M64
    return x - (1 << 64) if x >= (1 << 63) else x


_GOLDEN = _i64(0x9E3779B97F4A7C15)
_MIX1 = _i64(0xBF58476D1CE4E5B9)
_MIX2 = _i64(0x94D049BB133111EB)


def _srl(x: torch.Tensor, k: int) -> torch.Tensor:
    """Logical right shift of an int64 tensor (torch's >> is arithmetic)."""
    return (x >> k) & ((1 << (64 - k)) - 1)


def _finalise(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _srl(z, 30)) * _MIX1
    z = (z ^ _srl(z, 27)) * _MIX2
    return z ^ _srl(z, 31)


def splitmix64_int(x: int) -> int:
    """Scalar SplitMix64 finaliser on Python ints (used for keys and as the test reference)."""
    z = x & _M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


_STREAMS = {"latent": 1, "q": 2, "perm": 3, "len": 4, "outlier": 5, "append": 6, "misc": 7}


def stream_key(seed: int, stream: str) -> int:
    return _i64(splitmix64_int((seed * 0x9E3779B97F4A7C15 + _STREAMS[stream] * 0xD1B54A32D192ED03) & _M64))


def raw64(key: int, counters: torch.Tensor) -> torch.Tensor:
    """Counter-based SplitMix64: int64 tensor of raw 64-bit outputs for int64 counters."""
    return _finalise(key + (counters + 1) * _GOLDEN)


def uniform(key: int, counters: torch.Tensor) -> torch.Tensor:
    """Uniform doubles in the open interval (0, 1), 53 random bits each."""
    return _srl(raw64(key, counters), 11).to(torch.float64) * (2.0 ** -53) + 2.0 ** -54


def normal_pairs(key: int, pair_counters: torch.Tensor) -> torch.Tensor:
    """Box-Muller: for each pair counter c, two standard normals. Returns shape [..., 2] float64."""
    u1 = uniform(key, 2 * pair_counters)
    u2 = uniform(key, 2 * pair_counters + 1)
    r = torch.sqrt(-2.0 * torch.log(u1))
    th = (2.0 * math.pi) * u2
    return torch.stack((r * torch.cos(th), r * torch.sin(th)), dim=-1)


def seeded_perm(seed: int, stream: str, n: int) -> torch.Tensor:
    """A seeded permutation of range(n) (Fisher-Yates driven by the counter generator, on the host)."""
    key = stream_key(seed, stream)
    idx = torch.arange(n - 1, 0, -1, dtype=torch.int64)
    u = uniform(key, idx)
    j = torch.floor(u * (idx + 1).to(torch.float64)).to(torch.int64)
    perm = np.arange(n, dtype=np.int64)
    jj = j.numpy()
    for pos, i in enumerate(range(n - 1, 0, -1)):
        k = int(jj[pos])
        perm[i], perm[k] = perm[k], perm[i]
    return torch.from_numpy(perm)


def latent_fp8(seed: int, req: int, tok: torch.Tensor, outliers: list[int], device) -> torch.Tensor:
    """FP8 E4M3 bytes [len(tok), 576] of the latent of tokens `tok` of request `req`.

    Values are N(0, 1); the channels in `outliers` are multiplied by 20 before the cast.
    """
    key = stream_key(seed, "latent")
    tok = tok.to(device=device, dtype=torch.int64)
    base = ((req << 30) + tok) * (D_LATENT // 2)
    pc = base[:, None] + torch.arange(D_LATENT // 2, device=device, dtype=torch.int64)[None, :]
    x = normal_pairs(key, pc).reshape(tok.numel(), D_LATENT)
    if outliers:
        x[:, torch.tensor(outliers, device=device, dtype=torch.int64)] *= 20.0
    return x.to(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)


def query_bf16(seed: int, batch: int, heads: int, device) -> torch.Tensor:
    """Q [batch, heads, 576] in BF16, N(0, 1)."""
    key = stream_key(seed, "q")
    rh = torch.arange(batch * heads, device=device, dtype=torch.int64)
    pc = (rh * (D_LATENT // 2))[:, None] + torch.arange(D_LATENT // 2, device=device, dtype=torch.int64)[None, :]
    x = normal_pairs(key, pc).reshape(batch, heads, D_LATENT)
    return x.to(torch.float32).to(torch.bfloat16)


def draw_outliers(seed: int, count: int) -> list[int]:
    if count == 0:
        return []
    return sorted(int(c) for c in seeded_perm(seed, "outlier", D_LATENT)[:count])


@dataclass
class Workload:
    """One decode problem: queries, a paged FP8 latent pool and its CSR page table.

    kv_indptr / kv_indices follow the CSR convention of the pages' plan() call (The Smoking Gun,
    section "What Message 1408 Actually Reveals"): request r owns pages
    kv_indices[kv_indptr[r]:kv_indptr[r+1]], and token t of r sits at offset t % 64 of page t // 64.
    """
    name: str
    batch: int
    heads: int
    kv_len: np.ndarray            # int32 [B], tokens per request
    kv_indptr: np.ndarray         # int32 [B+1], in pages
    kv_indices: np.ndarray        # int32 [nnz], page ids
    num_pages: int                # pages in the pool
    sm_scale: float
    seed: int
    outliers: list
    q: torch.Tensor               # bf16 [B, H, 576]
    pool_fp8: torch.Tensor        # uint8 [num_pages, 64, 576], unowned slots = 0x7F (NaN)
    src_fp8: torch.Tensor         # uint8 [T, 576], every owned token, request-major
    slots: torch.Tensor           # int64 [T], slot = page * 64 + offset of each src row
    meta: dict = field(default_factory=dict)

    @property
    def total_tokens(self) -> int:
        return int(self.kv_len.sum())


def build_workload(name: str, lens, heads: int, pool_pages: int, seed: int = 0, outliers: int = 0,
                   device="cpu", extra_pages=None, sm_scale: float | None = None,
                   chunk_tokens: int = 1 << 16) -> Workload:
    """Draw a workload: requests of the given lengths, pages scattered over a pool of `pool_pages`.

    Pages come from a seeded permutation of the pool; request r takes the next ceil(L_r / 64)
    (+ extra_pages[r]) of it. Slots that no request's tokens fill stay 0x7F (FP8 NaN), so a kernel
    that reads past a length or through a wrong page id produces NaN.
    """
    lens = np.asarray(lens, dtype=np.int64)
    B = len(lens)
    need = (lens + PAGE - 1) // PAGE
    if extra_pages is not None:
        need = need + np.asarray(extra_pages, dtype=np.int64)
    if need.sum() > pool_pages:
        raise ValueError(f"{name}: {need.sum()} pages needed, pool has {pool_pages}")
    perm = seeded_perm(seed, "perm", pool_pages).numpy()
    indptr = np.zeros(B + 1, dtype=np.int64)
    indptr[1:] = np.cumsum(need)
    indices = perm[: indptr[-1]].astype(np.int32)
    outl = draw_outliers(seed, outliers)
    pool = torch.full((pool_pages, PAGE, D_LATENT), FP8_NAN, dtype=torch.uint8, device=device)
    flat = pool.view(pool_pages * PAGE, D_LATENT)
    T = int(lens.sum())
    src = torch.empty((T, D_LATENT), dtype=torch.uint8, device=device)
    slots = torch.empty((T,), dtype=torch.int64, device=device)
    idx_dev = torch.from_numpy(indices.astype(np.int64)).to(device)
    row = 0
    for r in range(B):
        L = int(lens[r])
        for t0 in range(0, L, chunk_tokens):
            t1 = min(L, t0 + chunk_tokens)
            tok = torch.arange(t0, t1, dtype=torch.int64, device=device)
            lat = latent_fp8(seed, r, tok, outl, device)
            pg = idx_dev[int(indptr[r]) + tok // PAGE]
            sl = pg * PAGE + tok % PAGE
            flat[sl] = lat
            src[row + t0: row + t1] = lat
            slots[row + t0: row + t1] = sl
        row += L
    q = query_bf16(seed, B, heads, device)
    return Workload(name=name, batch=B, heads=heads, kv_len=lens.astype(np.int32),
                    kv_indptr=indptr.astype(np.int32), kv_indices=indices, num_pages=pool_pages,
                    sm_scale=(1.0 / math.sqrt(192.0)) if sm_scale is None else sm_scale, seed=seed,
                    outliers=outl, q=q, pool_fp8=pool, src_fp8=src, slots=slots)


def log_uniform_lengths(seed: int, n: int, lo: int, hi: int, pool_tokens: int, fill: float = 0.9):
    """n lengths drawn log-uniform on [lo, hi], then scaled down (if needed) to fill at most
    `fill` of the pool, rounded, and clamped to >= 1 token."""
    u = uniform(stream_key(seed, "len"), torch.arange(n, dtype=torch.int64)).numpy()
    raw = np.exp(np.log(lo) + u * (np.log(hi) - np.log(lo)))
    f = min(1.0, fill * pool_tokens / raw.sum())
    return np.maximum(1, np.rint(raw * f)).astype(np.int64), raw


def append_tokens(w: Workload, device) -> tuple[torch.Tensor, torch.Tensor]:
    """The token each request appends at a decode step: its latent at index L_r, and the slot.

    The slot is offset L_r % 64 of page L_r // 64 of the request's page list (the page list must
    already have room: build the workload with one extra page where L_r is a multiple of 64).
    """
    outl = w.outliers
    src = torch.empty((w.batch, D_LATENT), dtype=torch.uint8, device=device)
    slots = torch.empty((w.batch,), dtype=torch.int64, device=device)
    for r in range(w.batch):
        L = int(w.kv_len[r])
        src[r] = latent_fp8(w.seed, r, torch.tensor([L], dtype=torch.int64), outl, device)[0]
        page = int(w.kv_indices[int(w.kv_indptr[r]) + L // PAGE])
        slots[r] = page * PAGE + L % PAGE
    return src, slots


# Named workloads: the five decode problems, by what they are and their sizes.
def workload(name: str, device="cpu", seed: int = 0) -> Workload:
    if name == "mla_tiny_b1_h16_l256":
        # batch 1, 16 heads, 256 tokens, 8-page pool, seeded page permutation
        return build_workload(name, [256], heads=16, pool_pages=8, seed=seed, device=device)
    if name == "mla_fp8_b44_h128_l32k":
        # 44 requests x 32768 tokens, 1.5 Mi-token pool, 4 outlier channels x20
        return build_workload(name, [32768] * 44, heads=128, pool_pages=(3 << 19) // PAGE,
                              seed=seed, outliers=4, device=device)
    if name == "mla_nvfp4_b10_h128_l160k":
        # 10 requests x 163840 tokens (+1 appended each step), 32768-page pool
        w = build_workload(name, [163840] * 10, heads=128, pool_pages=32768, seed=seed, outliers=4,
                           device=device, extra_pages=[1] * 10)
        return w
    if name == "mla_nvfp4_b1_h128_l1m":
        # one request of 1,048,576 tokens, its 16384 pages permuted within a 16384-page pool
        return build_workload(name, [1 << 20], heads=128, pool_pages=16384, seed=seed, outliers=4,
                              device=device)
    if name == "mla_fp8_mixed_b64_h128_pool495552":
        pool_tokens = 495552
        lens, raw = log_uniform_lengths(seed, 64, 512, 65536, pool_tokens)
        w = build_workload(name, lens, heads=128, pool_pages=pool_tokens // PAGE, seed=seed,
                           outliers=4, device=device)
        w.meta["raw_lengths"] = raw
        return w
    raise KeyError(name)


WORKLOADS = ["mla_tiny_b1_h16_l256", "mla_fp8_b44_h128_l32k", "mla_nvfp4_b10_h128_l160k",
             "mla_nvfp4_b1_h128_l1m", "mla_fp8_mixed_b64_h128_pool495552"]
