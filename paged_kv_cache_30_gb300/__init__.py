"""paged_kv_cache_30_gb300 -- split-KV paged decode attention for GB300 (sm_103a).

A thin ctypes binding over ``libpkv.so`` (the C ABI declared in
``include/pkv.h``).  Every function here only marshals arguments: the attention
itself runs in the library's CUDA kernels.  PyTorch provides device memory and
streams.  There is no CPU fallback: if the library is missing, importing the
entry points raises.

Names follow the C ABI without its ``pkv_`` prefix:

    paged_decode_attn(q, kv_cache, block_table, seq_lens, sinks, window, scale,
                      page_size, num_kv_splits, out, lse=None, stream=None)
    paged_decode_attn_noalloc(...)   same arguments; allocates nothing
    mla_verify_attn(q, latent_cache, block_table, seq_lens, real_seq_lens, qlen,
                    scale, page_size, k_scale, out, lse, num_kv_splits=0,
                    stream=None)
    gqa_kv_append(k, v, kv_cache, block_table, seq_lens, page_size, stream=None)
    mla_kv_append(latent, latent_cache, block_table, seq_lens, qlen, page_size,
                  k_scale=None, stream=None)
    num_kv_splits(max_seq_len, batch, qlen, num_heads, sm_count, ...)
    init(device, workspace_bytes=0), check_errors(device),
    check_counters(device), shutdown(), version()
"""
from __future__ import annotations

import ctypes
import os
import struct
import threading

__all__ = [
    "PkvError", "load_library", "library_path", "init", "paged_decode_attn",
    "paged_decode_attn_noalloc",
    "mla_verify_attn", "gqa_kv_append", "mla_kv_append", "num_kv_splits", "check_errors", "check_counters", "shutdown",
    "version", "last_error",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libpkv.so")

PKV_OK = 0
ERRORS = {
    -1: "PKV_ERR_INVALID_ARG", -2: "PKV_ERR_UNSUPPORTED", -3: "PKV_ERR_ALIGNMENT",
    -4: "PKV_ERR_WORKSPACE", -5: "PKV_ERR_CAPTURE", -6: "PKV_ERR_CUDA",
    -7: "PKV_ERR_BAD_BLOCK_TABLE",
}
DTYPE_BF16, DTYPE_F32, DTYPE_I32, DTYPE_FP8 = 1, 2, 3, 4


class PkvError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{ERRORS.get(code, code)}: {message}")
        self.code = code


class PkvTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 5), ("stride", ctypes.c_int64 * 5)]


assert ctypes.sizeof(PkvTensor) == 96


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _LIB_PATH


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libpkv.so (built by ``paged_kv_cache_30_gb300.build.build()``)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _LIB_PATH
        if not os.path.exists(p):
            raise ImportError(
                f"{p} is missing: build it with `python -c \"import __graft_entry__ as g; "
                f"g.build()\"` (nvcc, sm_103a); there is no fallback implementation")
        lib = ctypes.CDLL(p)
        T = ctypes.POINTER(PkvTensor)
        i32, f32, vp = ctypes.c_int, ctypes.c_float, ctypes.c_void_p
        lib.pkv_init.argtypes = [i32, ctypes.c_size_t]
        lib.pkv_paged_decode_attn.argtypes = [T, T, T, T, T, i32, f32, i32, i32, T, T, vp]
        lib.pkv_paged_decode_attn_noalloc.argtypes = [T, T, T, T, T, i32, f32, i32, i32, T, T, vp]
        lib.pkv_mla_verify_attn.argtypes = [T, T, T, T, T, i32, f32, i32, T, T, T, i32, vp]
        lib.pkv_mla_quantize_q.argtypes = [T, T, T, vp]
        lib.pkv_mla_verify_attn_fp8_native.argtypes = [T, T, T, T, T, T, i32, ctypes.c_float, i32, T,
                                                       T, T, i32, vp]
        lib.pkv_gqa_kv_append.argtypes = [T, T, T, T, T, i32, vp]
        lib.pkv_mla_kv_append.argtypes = [T, T, T, T, i32, i32, T, vp]
        lib.pkv_num_kv_splits.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.c_double, i32, i32]
        lib.pkv_check_errors.argtypes = [i32, ctypes.POINTER(ctypes.c_int32)]
        lib.pkv_check_counters.argtypes = [i32, ctypes.POINTER(ctypes.c_int64)]
        lib.pkv_selftest_wait_timeout.argtypes = [i32, vp]
        lib.pkv_last_error.restype = ctypes.c_char_p
        for name in ("pkv_init", "pkv_paged_decode_attn", "pkv_paged_decode_attn_noalloc",
                     "pkv_mla_verify_attn", "pkv_mla_quantize_q",
                     "pkv_mla_verify_attn_fp8_native", "pkv_gqa_kv_append", "pkv_mla_kv_append",
                     "pkv_num_kv_splits", "pkv_check_errors", "pkv_check_counters",
                     "pkv_selftest_wait_timeout",
                     "pkv_shutdown", "pkv_version"):
            getattr(lib, name).restype = i32
        if path is None:
            _lib = lib
        return lib


def last_error() -> str:
    return load_library().pkv_last_error().decode()


def _check(rc: int) -> int:
    if rc < 0:
        raise PkvError(rc, last_error())
    return rc


_DTYPES = None


def _dtype_code(t) -> int:
    global _DTYPES
    if _DTYPES is None:
        import torch
        _DTYPES = {torch.bfloat16: DTYPE_BF16, torch.float32: DTYPE_F32, torch.int32: DTYPE_I32,
                   torch.float8_e4m3fn: DTYPE_FP8}
    code = _DTYPES.get(t.dtype)
    if code is None:
        raise PkvError(-1, f"unsupported tensor dtype {t.dtype}")
    return code


_PACK = struct.Struct("<Qii5q5q")  # the byte layout of pkv_tensor (96 bytes)
_PAD = tuple((0,) * k for k in range(6))


def _desc(t):
    """pkv_tensor for a torch tensor (None -> NULL), packed in one call."""
    if t is None:
        return None
    n = t.dim()
    if n > 5:
        raise PkvError(-1, "tensors of more than 5 dims are not supported")
    pad = _PAD[5 - n]
    d = PkvTensor.from_buffer_copy(
        _PACK.pack(t.data_ptr(), _dtype_code(t), n, *t.shape, *pad, *t.stride(), *pad))
    return ctypes.byref(d)


def _stream(stream, device_tensor):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream(device_tensor.device).cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def init(device: int = 0, workspace_bytes: int = 0) -> None:
    _check(load_library().pkv_init(device, workspace_bytes))


def paged_decode_attn(q, kv_cache, block_table, seq_lens, sinks, window, scale, page_size,
                      num_kv_splits, out, lse=None, stream=None):
    """GQA paged decode attention (C: pkv_paged_decode_attn).  Writes ``out``
    (and ``lse`` if given) in place on ``stream`` (default: torch's current
    stream of q's device) and returns ``out``."""
    lib = load_library()
    _check(lib.pkv_paged_decode_attn(
        _desc(q), _desc(kv_cache), _desc(block_table), _desc(seq_lens), _desc(sinks),
        int(window or 0), float(scale), int(page_size), int(num_kv_splits), _desc(out),
        _desc(lse), _stream(stream, q)))
    return out


def paged_decode_attn_noalloc(q, kv_cache, block_table, seq_lens, sinks, window, scale,
                              page_size, num_kv_splits, out, lse=None, stream=None):
    """GQA paged decode attention that allocates nothing (C:
    pkv_paged_decode_attn_noalloc): for callers that cannot let a library
    allocate device memory.  Its scratch is a fixed array inside the library
    (batch x kv heads <= 4096, batch x kv heads x splits <= 2048); calls must
    not overlap on the GPU."""
    lib = load_library()
    _check(lib.pkv_paged_decode_attn_noalloc(
        _desc(q), _desc(kv_cache), _desc(block_table), _desc(seq_lens), _desc(sinks),
        int(window or 0), float(scale), int(page_size), int(num_kv_splits), _desc(out),
        _desc(lse), _stream(stream, q)))
    return out


def mla_verify_attn(q, latent_cache, block_table, seq_lens, real_seq_lens, qlen, scale,
                    page_size, k_scale, out, lse, num_kv_splits=0, stream=None):
    """MLA causal verify (C: pkv_mla_verify_attn).  ``k_scale`` is a device
    fp32 scalar tensor or None.  Writes ``out`` and ``lse`` in place."""
    lib = load_library()
    _check(lib.pkv_mla_verify_attn(
        _desc(q), _desc(latent_cache), _desc(block_table), _desc(seq_lens),
        _desc(real_seq_lens), int(qlen), float(scale), int(page_size), _desc(k_scale),
        _desc(out), _desc(lse), int(num_kv_splits), _stream(stream, q)))
    return out


def mla_quantize_q(q, q8, q_scale, stream=None):
    """Per-(row, head) e4m3 quantisation of an MLA query (C: pkv_mla_quantize_q):
    writes ``q8`` (float8_e4m3fn [R, 128, 576]) and ``q_scale`` (fp32 [R, 128])."""
    lib = load_library()
    _check(lib.pkv_mla_quantize_q(_desc(q), _desc(q8), _desc(q_scale), _stream(stream, q)))
    return q8, q_scale


def mla_verify_attn_fp8_native(q8, q_scale, latent_cache, block_table, seq_lens, real_seq_lens,
                               qlen, scale, page_size, k_scale, out, lse, num_kv_splits=0,
                               stream=None):
    """MLA causal verify over an e4m3 cache with an e4m3 query (C:
    pkv_mla_verify_attn_fp8_native).  Writes ``out`` and ``lse`` in place."""
    lib = load_library()
    _check(lib.pkv_mla_verify_attn_fp8_native(
        _desc(q8), _desc(q_scale), _desc(latent_cache), _desc(block_table), _desc(seq_lens),
        _desc(real_seq_lens), int(qlen), float(scale), int(page_size), _desc(k_scale),
        _desc(out), _desc(lse), int(num_kv_splits), _stream(stream, q8)))
    return out


def gqa_kv_append(k, v, kv_cache, block_table, seq_lens, page_size, stream=None):
    """Write each request's current token (position seq_lens[b] - 1) into the
    paged GQA cache in place (C: pkv_gqa_kv_append).  Returns ``kv_cache``."""
    lib = load_library()
    _check(lib.pkv_gqa_kv_append(_desc(k), _desc(v), _desc(kv_cache), _desc(block_table),
                                 _desc(seq_lens), int(page_size), _stream(stream, k)))
    return kv_cache


def mla_kv_append(latent, latent_cache, block_table, seq_lens, qlen, page_size, k_scale=None,
                  stream=None):
    """Write verify row t of request b (position seq_lens[b] - qlen + t) into
    the paged latent cache in place; an e4m3 cache stores e4m3(x / k_scale)
    (C: pkv_mla_kv_append).  Returns ``latent_cache``."""
    lib = load_library()
    _check(lib.pkv_mla_kv_append(_desc(latent), _desc(latent_cache), _desc(block_table),
                                 _desc(seq_lens), int(qlen), int(page_size), _desc(k_scale),
                                 _stream(stream, latent)))
    return latent_cache


def num_kv_splits(max_seq_len, batch, qlen, num_heads, sm_count, block_h=64, occupancy=1.0,
                  min_work_per_split=64, max_splits=8) -> int:
    """Static split cap, safe to bake into a CUDA graph (C: pkv_num_kv_splits)."""
    return _check(load_library().pkv_num_kv_splits(
        int(max_seq_len), int(batch), int(qlen), int(num_heads), int(sm_count), int(block_h),
        float(occupancy), int(min_work_per_split), int(max_splits)))


def check_errors(device: int = 0) -> int:
    """Read and clear the device error word; raises PkvError if a bit was set."""
    flags = ctypes.c_int32(0)
    rc = load_library().pkv_check_errors(device, ctypes.byref(flags))
    if rc < 0:
        raise PkvError(rc, last_error())
    return flags.value


def selftest_wait_timeout(device: int = 0, stream=None) -> None:
    """Failure-detection self-test (C: pkv_selftest_wait_timeout): a bounded
    wait that runs out (~1 s) and raises bit 4 of the device error word."""
    import torch
    s = stream if stream is not None else torch.cuda.current_stream(device)
    _check(load_library().pkv_selftest_wait_timeout(
        device, ctypes.c_void_p(s if isinstance(s, int) else s.cuda_stream)))


def check_counters(device: int = 0) -> int:
    n = ctypes.c_int64(0)
    _check(load_library().pkv_check_counters(device, ctypes.byref(n)))
    return n.value


def shutdown() -> None:
    _check(load_library().pkv_shutdown())


def version() -> int:
    return load_library().pkv_version()
