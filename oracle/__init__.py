"""fp64 CPU oracle for split-KV paged decode attention (ctypes wrapper).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product path (``paged_kv_cache_30_gb300``) never imports it and
shares no code with it; the two meet only through the seeded input
generators in ``paged_kv_cache_30_gb300.workloads``.

The arithmetic lives in ``pkv_oracle.c`` (plain C, fp64, one output row at a
time); this module only compiles it with gcc and marshals arrays.  Citations
of the pages each step follows are in the C file's header and functions.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libpkv_oracle.so")
_lock = threading.Lock()
_lib = None

# -ffp-contract=off: no fused multiply-add contraction, so the same source gives
# the same bits on x86-64 and aarch64.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off"]


def compile_oracle(src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile an oracle source file into a shared library; returns its path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build() -> str:
    """(Re)build the oracle library if the source is newer than the binary."""
    if (not os.path.exists(_LIB_PATH)
            or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        compile_oracle()
    return _LIB_PATH


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
    lib.pkv_oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.pkv_oracle_bf16_to_f64.restype = dbl
    lib.pkv_oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
    lib.pkv_oracle_e4m3_to_f64.restype = dbl
    lib.pkv_oracle_gqa_decode.argtypes = [
        vp, i64, i64,            # q, strides
        vp, i64, i64, i64, i64,  # kv, strides, num_blocks
        vp, i64, i64,            # block table, stride, max_blocks
        vp, vp,                  # seq_lens, sinks
        i32, dbl, i32,           # window, scale, page_size
        i32, i32, i32, i32,      # B, Hq, Hkv, D
        vp, i64, vp, vp, i32]    # rows, nrows, out, lse, nthreads
    lib.pkv_oracle_gqa_decode.restype = i32
    lib.pkv_oracle_mla_verify.argtypes = [
        vp, i64, i64,            # q, strides
        vp, i32, i64, i64, i64,  # cache, fp8, strides, num_pages
        vp, i64, i64,            # block table, stride, max_blocks
        vp, vp,                  # seq_lens, real_seq_lens
        i32, dbl, i32, dbl,      # qlen, scale, page_size, k_scale
        i32, i32, i32, i32,      # B, H, Lk, Lv
        vp, i64, vp, vp, i32]    # rows, nrows, out, lse, nthreads
    lib.pkv_oracle_mla_verify.restype = i32
    lib.pkv_oracle_mla_verify_q8.argtypes = [
        vp, i64, i64, vp, i64,   # q8 codes, strides, q scales, row stride
        vp, i32, i64, i64, i64,  # cache, fp8, strides, num_pages
        vp, i64, i64,            # block table, stride, max_blocks
        vp, vp,                  # seq_lens, real_seq_lens
        i32, dbl, i32, dbl,      # qlen, scale, page_size, k_scale
        i32, i32, i32, i32,      # B, H, Lk, Lv
        vp, i64, vp, vp, i32]    # rows, nrows, out, lse, nthreads
    lib.pkv_oracle_mla_verify_q8.restype = i32
    lib.pkv_oracle_mla_quantize_q.argtypes = [vp, i64, i64, i32, i32, i32, vp, vp]
    lib.pkv_oracle_mla_quantize_q.restype = i32
    lib.pkv_oracle_f32_to_e4m3.restype = ctypes.c_uint8
    lib.pkv_oracle_f32_to_e4m3.argtypes = [ctypes.c_float]
    i64, vp, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    lib.pkv_oracle_gqa_kv_append.argtypes = [vp, vp, i64, i64, vp, i64, i64, i64, i64, vp, i64,
                                             i64, vp, ci, i64, i64, i64, ctypes.POINTER(i64)]
    lib.pkv_oracle_mla_kv_append.argtypes = [vp, i64, vp, ci, i64, i64, i64, vp, i64, i64, vp, ci,
                                             ci, ctypes.c_float, i64, i64, ctypes.POINTER(i64)]
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the oracle library (building it first if needed).  With ``path``,
    load that library instead (used by the mutation tests)."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
    return _lib


def _np(t, dtype):
    """A C-contiguous numpy view/copy of a CPU torch tensor or numpy array."""
    if t is None:
        return None
    if hasattr(t, "detach"):
        import torch
        t = t.detach().cpu()
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16)
        elif t.dtype == getattr(torch, "float8_e4m3fn", None):
            t = t.view(torch.uint8)
        t = t.numpy()
    return np.ascontiguousarray(t).view(dtype) if t.dtype.itemsize == np.dtype(dtype).itemsize \
        else np.ascontiguousarray(t.astype(dtype))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _threads(nthreads):
    return nthreads if nthreads else (os.cpu_count() or 1)


def bf16_to_f64(bits: int, lib=None) -> float:
    return (lib or load()).pkv_oracle_bf16_to_f64(bits & 0xFFFF)


def e4m3_to_f64(bits: int, lib=None) -> float:
    return (lib or load()).pkv_oracle_e4m3_to_f64(bits & 0xFF)


class OracleError(RuntimeError):
    pass


def gqa_decode(q, kv_cache, block_table, seq_lens, sinks, window, scale, page_size,
               rows=None, nthreads=None, lib=None):
    """fp64 GQA paged decode.

    q: [B, Hq, D] bf16; kv_cache: [num_blocks, Hkv, P, 2D] bf16 (contiguous);
    block_table: [B, max_blocks] int32; seq_lens: [B] int32; sinks: [Hq] fp32 or
    None; window: int (<= 0: none); scale: python float (rounded to fp32 first,
    as the library receives it).  rows: optional 1-D array of b*Hq + h indices.
    Returns (out [nrows, D] float64, lse [nrows] float64).
    """
    lib = lib or load()
    qn = _np(q, np.uint16)
    kvn = _np(kv_cache, np.uint16)
    btn = _np(block_table, np.int32)
    sln = _np(seq_lens, np.int32)
    snk = _np(sinks, np.float32)
    B, Hq, D = qn.shape
    nb, Hkv, P, D2 = kvn.shape
    assert D2 == 2 * D and P == page_size
    rws = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    nrows = B * Hq if rws is None else rws.shape[0]
    out = np.zeros((nrows, D), dtype=np.float64)
    lse = np.zeros((nrows,), dtype=np.float64)
    rc = lib.pkv_oracle_gqa_decode(
        _ptr(qn), Hq * D, D,
        _ptr(kvn), Hkv * P * D2, P * D2, D2, nb,
        _ptr(btn), btn.shape[1], btn.shape[1],
        _ptr(sln), _ptr(snk),
        int(window or 0), float(np.float32(scale)), int(page_size),
        B, Hq, Hkv, D,
        _ptr(rws), nrows, _ptr(out), _ptr(lse), _threads(nthreads))
    if rc != 0:
        raise OracleError(f"pkv_oracle_gqa_decode failed with status {rc}")
    return out, lse


def mla_verify(q, latent_cache, block_table, seq_lens, real_seq_lens, qlen, scale,
               page_size, k_scale=None, Lv=512, rows=None, nthreads=None, lib=None):
    """fp64 MLA causal verify.

    q: [B*qlen, H, Lk] bf16; latent_cache: [num_pages, P, 1, Lk] (or
    [num_pages*P, 1, Lk]) bf16 or float8_e4m3fn; k_scale: python float or None
    (1.0; ignored for bf16).  Returns (out [nrows, Lv], lse [nrows]) in float64.
    """
    import torch
    lib = lib or load()
    fp8 = int(latent_cache.dtype == torch.float8_e4m3fn)
    qn = _np(q, np.uint16)
    cn = _np(latent_cache, np.uint8 if fp8 else np.uint16)
    btn = _np(block_table, np.int32)
    sln = _np(seq_lens, np.int32)
    rln = _np(real_seq_lens, np.int32)
    R, H, Lk = qn.shape
    assert R % qlen == 0
    B = R // qlen
    if cn.ndim == 3:
        cn = cn.reshape(-1, page_size, 1, Lk)
    num_pages, P, one, Lk2 = cn.shape
    assert one == 1 and Lk2 == Lk and P == page_size
    rws = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    nrows = R * H if rws is None else rws.shape[0]
    out = np.zeros((nrows, Lv), dtype=np.float64)
    lse = np.zeros((nrows,), dtype=np.float64)
    ks = 1.0 if (k_scale is None or not fp8) else float(np.float32(k_scale))
    rc = lib.pkv_oracle_mla_verify(
        _ptr(qn), H * Lk, Lk,
        _ptr(cn), fp8, P * Lk, Lk, num_pages,
        _ptr(btn), btn.shape[1], btn.shape[1],
        _ptr(sln), _ptr(rln),
        int(qlen), float(np.float32(scale)), int(page_size), ks,
        B, H, Lk, Lv,
        _ptr(rws), nrows, _ptr(out), _ptr(lse), _threads(nthreads))
    if rc != 0:
        raise OracleError(f"pkv_oracle_mla_verify failed with status {rc}")
    return out, lse


def mla_quantize_q(q, lib=None):
    """Per-(row, head) e4m3 quantisation of an MLA query [R, H, Lk] bf16:
    scale = absmax / 448 (fp32), code = e4m3(q / scale) with the quotient in
    fp32.  Returns (codes uint8 [R, H, Lk], scales float32 [R, H])."""
    lib = lib or load()
    qn = _np(q, np.uint16)
    R, H, Lk = qn.shape
    codes = np.zeros((R, H, Lk), dtype=np.uint8)
    scales = np.zeros((R, H), dtype=np.float32)
    rc = lib.pkv_oracle_mla_quantize_q(_ptr(qn), H * Lk, Lk, R, H, Lk, _ptr(codes), _ptr(scales))
    if rc != 0:
        raise OracleError(f"pkv_oracle_mla_quantize_q failed with status {rc}")
    return codes, scales


def mla_verify_q8(q8, q_scale, latent_cache, block_table, seq_lens, real_seq_lens, qlen, scale,
                  page_size, k_scale=None, Lv=512, rows=None, nthreads=None, lib=None):
    """mla_verify with the query given as e4m3 codes [B*qlen, H, Lk] (uint8)
    and per-(row, head) fp32 scales [B*qlen, H]: query = code value x scale."""
    import torch
    lib = lib or load()
    fp8 = int(latent_cache.dtype == torch.float8_e4m3fn)
    qn = np.ascontiguousarray(np.asarray(q8, dtype=np.uint8))
    qs = np.ascontiguousarray(np.asarray(q_scale, dtype=np.float32))
    cn = _np(latent_cache, np.uint8 if fp8 else np.uint16)
    btn = _np(block_table, np.int32)
    sln = _np(seq_lens, np.int32)
    rln = _np(real_seq_lens, np.int32)
    R, H, Lk = qn.shape
    assert R % qlen == 0 and qs.shape == (R, H)
    B = R // qlen
    if cn.ndim == 3:
        cn = cn.reshape(-1, page_size, 1, Lk)
    num_pages, P, one, Lk2 = cn.shape
    assert one == 1 and Lk2 == Lk and P == page_size
    rws = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    nrows = R * H if rws is None else rws.shape[0]
    out = np.zeros((nrows, Lv), dtype=np.float64)
    lse = np.zeros((nrows,), dtype=np.float64)
    ks = 1.0 if (k_scale is None or not fp8) else float(np.float32(k_scale))
    rc = lib.pkv_oracle_mla_verify_q8(
        _ptr(qn), H * Lk, Lk, _ptr(qs), H,
        _ptr(cn), fp8, P * Lk, Lk, num_pages,
        _ptr(btn), btn.shape[1], btn.shape[1],
        _ptr(sln), _ptr(rln),
        int(qlen), float(np.float32(scale)), int(page_size), ks,
        B, H, Lk, Lv,
        _ptr(rws), nrows, _ptr(out), _ptr(lse), _threads(nthreads))
    if rc != 0:
        raise OracleError(f"pkv_oracle_mla_verify_q8 failed with status {rc}")
    return out, lse


def f32_to_e4m3(x: float, lib=None) -> int:
    """e4m3 'fn' code of an fp32 value: nearest, ties to even, saturating at 448."""
    return (lib or load()).pkv_oracle_f32_to_e4m3(float(np.float32(x)))


def gqa_kv_append(k, v, kv_cache, block_table, seq_lens, page_size, lib=None):
    """Write each request's current token (position seq_lens[b] - 1) into a
    copy of the GQA cache.  k, v: [B, Hkv, D] bf16; kv_cache: [num_blocks, Hkv,
    P, 2D] bf16.  Returns (new cache as uint16 numpy array, rows skipped)."""
    lib = lib or load()
    kn, vn = _np(k, np.uint16), _np(v, np.uint16)
    cache = _np(kv_cache, np.uint16).copy()
    btn, sln = _np(block_table, np.int32), _np(seq_lens, np.int32)
    B, Hkv, D = kn.shape
    nb, Hkv2, P, D2 = cache.shape
    assert Hkv2 == Hkv and D2 == 2 * D and P == page_size
    skipped = ctypes.c_int64(0)
    rc = lib.pkv_oracle_gqa_kv_append(_ptr(kn), _ptr(vn), Hkv * D, D, _ptr(cache), Hkv * P * D2,
                                      P * D2, D2, nb, _ptr(btn), btn.shape[1], btn.shape[1],
                                      _ptr(sln), int(page_size), B, Hkv, D, ctypes.byref(skipped))
    if rc != 0:
        raise OracleError(f"pkv_oracle_gqa_kv_append failed with status {rc}")
    return cache, skipped.value


def mla_kv_append(latent, latent_cache, block_table, seq_lens, qlen, page_size, k_scale=None,
                  lib=None):
    """Write verify row t of request b (position seq_lens[b] - qlen + t) into a
    copy of the latent cache.  latent: [B*qlen, Lk] bf16; latent_cache:
    [num_pages, P, 1, Lk] bf16 or float8_e4m3fn.  Returns (new cache as a
    uint16 / uint8 numpy array, rows skipped)."""
    import torch
    lib = lib or load()
    fp8 = int(latent_cache.dtype == torch.float8_e4m3fn)
    ln = _np(latent, np.uint16)
    cache = _np(latent_cache, np.uint8 if fp8 else np.uint16).copy()
    btn, sln = _np(block_table, np.int32), _np(seq_lens, np.int32)
    R, Lk = ln.shape
    assert R % qlen == 0
    num_pages, P, one, Lk2 = cache.shape
    assert one == 1 and Lk2 == Lk and P == page_size
    ks = 1.0 if (k_scale is None or not fp8) else float(np.float32(k_scale))
    skipped = ctypes.c_int64(0)
    rc = lib.pkv_oracle_mla_kv_append(_ptr(ln), Lk, _ptr(cache), fp8, P * Lk, Lk, num_pages,
                                      _ptr(btn), btn.shape[1], btn.shape[1], _ptr(sln), int(qlen),
                                      int(page_size), ks, R // qlen, Lk, ctypes.byref(skipped))
    if rc != 0:
        raise OracleError(f"pkv_oracle_mla_kv_append failed with status {rc}")
    return cache, skipped.value
