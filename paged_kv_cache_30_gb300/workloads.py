"""Seeded synthetic inputs for paged decode attention.

This module draws values, lengths and page assignments and lays them out in the
cache layouts the library reads.  It holds none of the attention arithmetic,
so both the CUDA library's callers and the CPU oracle can be fed from it
without sharing anything else.

Workload shapes follow the pages' problems (see the config builders at the end):
the Flint GQA decode layout (HND pages of 16 tokens x [K | V], GQA 8,
head_dim 128), the MLA verify layout (one 576-wide latent head, V = K[..., :512]),
and the block-table example of the transformers "Atencion paginada" page.

Recipe (all seeded, all CPU, deterministic for a given seed):
  * values: bf16 rounded from N(0, 1) float32 draws (numpy PCG64, drawn in
    fixed 4 Mi-element chunks with spawned child seeds, so the result does not
    depend on the thread count);
  * lengths: uniform integers, log-uniform round(exp(U(0, ln hi))) clamped to
    [lo, hi], or a constant;
  * block tables: each request receives distinct physical pages taken in order
    from one seeded permutation of the pool; unused entries are -1;
  * pool size: given, else ceil(1.25 * total pages needed);
  * FP8: N(0, 1) / k_scale clamped to +-448 and rounded to float8_e4m3fn.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

_CHUNK = 1 << 22


def _fill_normal(out_flat: torch.Tensor, seed: int, scale: float = 1.0,
                 fp8: bool = False) -> None:
    """Fill a flat CPU tensor (bf16 or float8_e4m3fn) with N(0,1)*scale draws."""
    n = out_flat.numel()
    nchunks = max(1, (n + _CHUNK - 1) // _CHUNK)
    seeds = np.random.SeedSequence(seed).spawn(nchunks)

    def work(i):
        lo = i * _CHUNK
        hi = min(n, lo + _CHUNK)
        g = np.random.Generator(np.random.PCG64(seeds[i]))
        x = g.standard_normal(hi - lo, dtype=np.float32)
        if scale != 1.0:
            x *= np.float32(scale)
        t = torch.from_numpy(x)
        if fp8:
            t = t.clamp_(-448.0, 448.0)
        out_flat[lo:hi].copy_(t.to(out_flat.dtype))

    workers = min(nchunks, os.cpu_count() or 1, 32)
    if workers <= 1:
        for i in range(nchunks):
            work(i)
    else:
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(work, range(nchunks)))


def normal(shape, seed: int, dtype=torch.bfloat16, scale: float = 1.0) -> torch.Tensor:
    """A CPU tensor of N(0,1)*scale values rounded to ``dtype``."""
    t = torch.empty(shape, dtype=dtype)
    _fill_normal(t.view(-1), seed, scale, fp8=(dtype == torch.float8_e4m3fn))
    return t


def draw_lengths(rng: np.random.Generator, B: int, kind: str, lo: int, hi: int) -> np.ndarray:
    if kind == "uniform":
        L = rng.integers(lo, hi + 1, size=B)
    elif kind == "loguniform":
        L = np.rint(np.exp(rng.uniform(0.0, math.log(hi), size=B)))
        L = np.clip(L, lo, hi)
    elif kind == "const":
        L = np.full(B, hi)
    else:
        raise ValueError(kind)
    return L.astype(np.int32)


def draw_block_table(rng: np.random.Generator, pages_needed: np.ndarray, max_blocks: int,
                     pool_pages: int | None) -> tuple[np.ndarray, int]:
    """Distinct physical pages per request from one seeded permutation of the pool."""
    total = int(pages_needed.sum())
    if pool_pages is None:
        pool_pages = max(1, math.ceil(1.25 * total))
    if total > pool_pages:
        raise ValueError(f"pool of {pool_pages} pages cannot hold {total}")
    perm = rng.permutation(pool_pages).astype(np.int32)
    bt = np.full((len(pages_needed), max_blocks), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(pages_needed):
        bt[b, :n] = perm[off:off + n]
        off += n
    return bt, pool_pages


@dataclass
class GQAProblem:
    q: torch.Tensor            # [B, Hq, D] bf16
    kv_cache: torch.Tensor     # [num_blocks, Hkv, P, 2D] bf16
    block_table: torch.Tensor  # [B, max_blocks] int32, -1 padded
    seq_lens: torch.Tensor     # [B] int32 (attended keys, current token included)
    sinks: torch.Tensor | None  # [Hq] fp32
    window: int
    scale: float
    page_size: int
    num_kv_splits: int = 0
    name: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def B(self):
        return self.q.shape[0]

    def attended_tokens(self) -> np.ndarray:
        L = self.seq_lens.numpy().astype(np.int64)
        if self.window > 0:
            return np.minimum(L, self.window)
        return L

    def kv_bytes(self) -> int:
        """Algorithmic KV bytes: attended tokens x Hkv x (K + V) x 2 bytes."""
        Hkv, D2 = self.kv_cache.shape[1], self.kv_cache.shape[3]
        return int(self.attended_tokens().sum()) * Hkv * D2 * 2


def gqa_problem(seed: int, B: int, Hq: int, Hkv: int, page_size: int, lengths: str,
                Lmin: int, Lmax: int, D: int = 128, pool_pages: int | None = None,
                sinks: bool = False, window: int = 0, scale: float | None = None,
                max_blocks: int | None = None, num_kv_splits: int = 0,
                seq_lens: np.ndarray | None = None, poison_unused: bool = False,
                name: str = "") -> GQAProblem:
    rng = np.random.default_rng(seed)
    L = draw_lengths(rng, B, lengths, Lmin, Lmax) if seq_lens is None \
        else np.asarray(seq_lens, dtype=np.int32)
    P = page_size
    if max_blocks is None:
        max_blocks = max(1, (Lmax + P - 1) // P)
    need = (L.astype(np.int64) + P - 1) // P
    bt, pool = draw_block_table(rng, need, max_blocks, pool_pages)
    q = normal((B, Hq, D), seed * 7919 + 1)
    kv = normal((pool, Hkv, P, 2 * D), seed * 7919 + 2)
    if poison_unused:
        used = np.zeros(pool, dtype=bool)
        used[bt[bt >= 0]] = True
        kv[torch.from_numpy(~used)] = float("nan")
        # slots past the last attended key of each request's last page
        for b in range(B):
            if L[b] > 0 and L[b] % P:
                kv[int(bt[b, (L[b] - 1) // P]), :, L[b] % P:, :] = float("nan")
            if window > 0 and L[b] > window:
                s = L[b] - window
                if s % P:
                    kv[int(bt[b, s // P]), :, : s % P, :] = float("nan")
                for p in range(s // P):
                    kv[int(bt[b, p])] = float("nan")
    snk = normal((Hq,), seed * 7919 + 3, dtype=torch.float32) if sinks else None
    return GQAProblem(
        q=q, kv_cache=kv, block_table=torch.from_numpy(bt), seq_lens=torch.from_numpy(L),
        sinks=snk, window=window, scale=(1.0 / math.sqrt(D)) if scale is None else scale,
        page_size=P, num_kv_splits=num_kv_splits, name=name,
        meta=dict(seed=seed, pool_pages=pool))


@dataclass
class MLAProblem:
    q: torch.Tensor             # [B*qlen, H, Lk] bf16
    latent_cache: torch.Tensor  # [num_pages, P, 1, Lk] bf16 or float8_e4m3fn
    block_table: torch.Tensor
    seq_lens: torch.Tensor
    real_seq_lens: torch.Tensor | None
    qlen: int
    scale: float
    page_size: int
    k_scale: float | None
    Lv: int = 512
    num_kv_splits: int = 0
    name: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def B(self):
        return self.seq_lens.shape[0]

    def kv_bytes(self) -> int:
        """Algorithmic latent bytes, a measurement convention: each request's
        keys min(L, L_real) read once x Lk x element size (V is part of K and
        is not counted twice)."""
        L = self.seq_lens.numpy().astype(np.int64)
        if self.real_seq_lens is not None:
            L = np.minimum(L, self.real_seq_lens.numpy().astype(np.int64))
        esz = self.latent_cache.element_size()
        return int(np.maximum(L, 0).sum()) * self.latent_cache.shape[-1] * esz


def mla_problem(seed: int, B: int, qlen: int, H: int, page_size: int, lengths: str,
                Lmin: int, Lmax: int, Lk: int = 576, Lv: int = 512, real_drop: int = 0,
                fp8: bool = False, k_scale: float = 0.05, scale: float | None = None,
                pool_pages: int | None = None, max_blocks: int | None = None,
                num_kv_splits: int = 0, seq_lens: np.ndarray | None = None,
                has_real: bool = True, name: str = "") -> MLAProblem:
    rng = np.random.default_rng(seed)
    L = draw_lengths(rng, B, lengths, Lmin, Lmax) if seq_lens is None \
        else np.asarray(seq_lens, dtype=np.int32)
    real = None
    if has_real:
        r = rng.integers(0, real_drop + 1, size=B) if real_drop > 0 else np.zeros(B, np.int64)
        real = torch.from_numpy(np.maximum(L - r, 0).astype(np.int32))
    P = page_size
    if max_blocks is None:
        max_blocks = max(1, (Lmax + P - 1) // P)
    need = (L.astype(np.int64) + P - 1) // P
    bt, pool = draw_block_table(rng, need, max_blocks, pool_pages)
    q = normal((B * qlen, H, Lk), seed * 7919 + 11)
    if fp8:
        cache = normal((pool, P, 1, Lk), seed * 7919 + 12, dtype=torch.float8_e4m3fn,
                       scale=1.0 / k_scale)
    else:
        cache = normal((pool, P, 1, Lk), seed * 7919 + 12)
    return MLAProblem(
        q=q, latent_cache=cache, block_table=torch.from_numpy(bt),
        seq_lens=torch.from_numpy(L), real_seq_lens=real, qlen=qlen,
        scale=(1.0 / math.sqrt(192)) if scale is None else scale, page_size=P,
        k_scale=k_scale if fp8 else None, Lv=Lv, num_kv_splits=num_kv_splits, name=name,
        meta=dict(seed=seed, pool_pages=pool))


# --------------------------------------------------------------------------
# The five workloads (shapes of the pages' problems).
# --------------------------------------------------------------------------

def tiny_gqa(seed: int = 0) -> GQAProblem:
    """B=4, Hq=8, Hkv=1, d=128, page 16, L ~ U[1,300], 128-page pool, cap 4."""
    return gqa_problem(seed, B=4, Hq=8, Hkv=1, page_size=16, lengths="uniform",
                       Lmin=1, Lmax=300, pool_pages=128, num_kv_splits=4,
                       name="tiny_gqa_b4")


def flint_gqa(seed: int = 0, window: int = 0, B: int = 64) -> GQAProblem:
    """B=64, Hq=64, Hkv=8, page 16 HND, log-uniform L in [1,32768], sinks; full
    attention (window 0) or sliding window 128."""
    return gqa_problem(seed, B=B, Hq=64, Hkv=8, page_size=16, lengths="loguniform",
                       Lmin=1, Lmax=32768, sinks=True, window=window,
                       name=f"flint_gqa_b{B}_{'w%d' % window if window else 'full'}")


def long_context(seed: int = 0, B: int = 1, num_kv_splits: int = 0) -> GQAProblem:
    """B in {1,8}, Hq=64, Hkv=8, page 32, L=131072, 40960-page pool."""
    return gqa_problem(seed, B=B, Hq=64, Hkv=8, page_size=32, lengths="const",
                       Lmin=131072, Lmax=131072, pool_pages=40960,
                       num_kv_splits=num_kv_splits, name=f"long_ctx_b{B}")


def mla_verify(seed: int = 0) -> MLAProblem:
    """B=32, qlen=4, H=128, Lk=576, Lv=512, page 16, L ~ U[512,8192],
    real = L - U[0,3], scale 1/sqrt(192), cap 8."""
    return mla_problem(seed, B=32, qlen=4, H=128, page_size=16, lengths="uniform",
                       Lmin=512, Lmax=8192, real_drop=3, num_kv_splits=8,
                       name="mla_verify_b32_q4")


def mla_fp8(seed: int = 0, k_scale: float = 0.05) -> MLAProblem:
    """B=128, qlen=1, H=128, FP8 e4m3 latent with scalar k_scale, page 16,
    log-uniform L in [1,32768], cap 16."""
    return mla_problem(seed, B=128, qlen=1, H=128, page_size=16, lengths="loguniform",
                       Lmin=1, Lmax=32768, fp8=True, k_scale=k_scale, has_real=False,
                       num_kv_splits=16, name="mla_fp8_b128")
