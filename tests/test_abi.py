"""CPU-side checks of the C ABI: the library loads, exports every entry point
declared in include/pkv.h, rejects bad arguments before touching a GPU, and
its host-only split-cap heuristic follows the verify page's contract."""
import ctypes
import os
import re

import pytest

import paged_kv_cache_30_gb300 as pkv
from paged_kv_cache_30_gb300 import build as pkv_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


@pytest.fixture(scope="module")
def lib():
    pkv_build.build()
    return pkv.load_library()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"PKV_API\s+[\w\s\*]+?\b(pkv_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_symbols()
    for n in ("pkv_paged_decode_attn", "pkv_mla_verify_attn", "pkv_init", "pkv_num_kv_splits",
              "pkv_check_errors", "pkv_check_counters", "pkv_last_error", "pkv_shutdown",
              "pkv_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), f"{name} is declared in pkv.h but not exported"


def test_version(lib):
    assert pkv.version() >= 100


def _t(shape, dtype, strides=None, ptr=0x10000):
    d = pkv.PkvTensor()
    d.data = ptr
    d.dtype = dtype
    d.ndim = len(shape)
    if strides is None:
        strides, acc = [], 1
        for s in reversed(shape):
            strides.insert(0, acc)
            acc *= s
    for i, (s, st) in enumerate(zip(shape, strides)):
        d.shape[i] = s
        d.stride[i] = st
    return d


# Fake device addresses, far enough apart that no two default views overlap
# (validation happens before any CUDA call, so nothing is dereferenced).
PTR = dict(q=0x1000000, kv=0x2000000, bt=0x8000000, sl=0x9000000, out=0xa000000,
           lse=0xb000000, sinks=0xc000000)


def _gqa_args(B=2, Hq=16, Hkv=2, D=128, P=16, nb=64, maxb=8):
    return dict(
        q=_t([B, Hq, D], pkv.DTYPE_BF16, ptr=PTR["q"]),
        kv=_t([nb, Hkv, P, 2 * D], pkv.DTYPE_BF16, ptr=PTR["kv"]),
        bt=_t([B, maxb], pkv.DTYPE_I32, ptr=PTR["bt"]), sl=_t([B], pkv.DTYPE_I32, ptr=PTR["sl"]),
        out=_t([B, Hq, D], pkv.DTYPE_BF16, ptr=PTR["out"]),
        lse=_t([B, Hq], pkv.DTYPE_F32, ptr=PTR["lse"]))


def _call(lib, a, sinks=None, window=0, scale=0.088, P=16, cap=0):
    r = ctypes.byref
    return lib.pkv_paged_decode_attn(r(a["q"]), r(a["kv"]), r(a["bt"]), r(a["sl"]),
                                     r(sinks) if sinks is not None else None, window, scale, P,
                                     cap, r(a["out"]), r(a["lse"]), None)


@pytest.mark.parametrize("mutate,code", [
    (lambda a: a.update(q=_t([2, 16, 64], pkv.DTYPE_BF16)), -2),               # head dim 64
    (lambda a: a.update(q=_t([2, 12, 128], pkv.DTYPE_BF16)), -2),              # Hq != 8 Hkv
    (lambda a: a.update(kv=_t([64, 2, 8, 256], pkv.DTYPE_BF16)), -1),          # P mismatch
    (lambda a: a.update(q=_t([2, 16, 128], pkv.DTYPE_F32)), -1),               # dtype
    (lambda a: a.update(bt=_t([3, 8], pkv.DTYPE_I32)), -1),                    # batch mismatch
    (lambda a: a.update(q=_t([2, 16, 128], pkv.DTYPE_BF16, ptr=PTR["q"] + 8)), -3),  # alignment
    (lambda a: a.update(kv=_t([64, 2, 16, 256], pkv.DTYPE_BF16, [8196, 4098, 256, 1],
                              ptr=PTR["kv"])), -3),
    (lambda a: a.update(kv=_t([64, 2, 16, 256], pkv.DTYPE_BF16, [8192, 4096, 512, 1],
                              ptr=PTR["kv"])), -1),
    (lambda a: a.update(q=_t([4096, 16, 128], pkv.DTYPE_BF16),
                        bt=_t([4096, 8], pkv.DTYPE_I32), sl=_t([4096], pkv.DTYPE_I32),
                        out=_t([4096, 16, 128], pkv.DTYPE_BF16),
                        lse=_t([4096, 16], pkv.DTYPE_F32)), -2),               # batch > 2048
    # outputs sharing memory with an input or with each other
    (lambda a: a.update(out=_t([2, 16, 128], pkv.DTYPE_BF16, ptr=PTR["q"])), -1),
    (lambda a: a.update(out=_t([2, 16, 128], pkv.DTYPE_BF16, ptr=PTR["q"] + 4096)), -1),
    (lambda a: a.update(lse=_t([2, 16], pkv.DTYPE_F32, ptr=PTR["out"] + 64)), -1),
    (lambda a: a.update(lse=_t([2, 16], pkv.DTYPE_F32, ptr=PTR["kv"] + 1024)), -1),
    (lambda a: a.update(out=_t([2, 16, 128], pkv.DTYPE_BF16, ptr=PTR["bt"])), -1),
    # block-table width x page size must stay below 2^31
    (lambda a: a.update(bt=_t([2, 1 << 27], pkv.DTYPE_I32, ptr=PTR["bt"])), -1),
])
def test_gqa_validation_rejects_before_any_cuda_call(lib, mutate, code):
    a = _gqa_args()
    mutate(a)
    assert _call(lib, a) == code
    assert pkv.last_error()


def test_gqa_validation_page_size_and_args(lib):
    a = _gqa_args()
    assert _call(lib, a, P=8) == -2
    assert _call(lib, a, cap=-1) == -1
    assert _call(lib, a, scale=float("inf")) == -1
    bad_sinks = _t([8], pkv.DTYPE_F32)
    assert _call(lib, a, sinks=bad_sinks) == -1
    r = ctypes.byref
    assert lib.pkv_paged_decode_attn(None, r(a["kv"]), r(a["bt"]), r(a["sl"]), None, 0, 1.0,
                                     16, 0, r(a["out"]), None, None) == -1


def test_gqa_outputs_adjacent_to_inputs_are_accepted_by_validation(lib):
    """out ending exactly where q begins is not an overlap: validation passes,
    and the call fails only later, at the first CUDA call (no GPU here)."""
    a = _gqa_args()
    q_bytes = 2 * 16 * 128 * 2
    a["out"] = _t([2, 16, 128], pkv.DTYPE_BF16, ptr=PTR["q"] - q_bytes)
    rc = _call(lib, a)
    assert rc != -1 or "overlaps" not in pkv.last_error()


def test_gqa_empty_batch_is_a_no_op(lib):
    a = _gqa_args(B=0)
    assert _call(lib, a) == 0


# ---------------------------------------------------- split-cap heuristic --
# Contract ("vllm.v1.attention.ops.triton_decode_attention", verify_num_kv_splits):
# programs per split = batch x row blocks; if they fit one round of
# occupancy x SMs slots, use slots // programs; otherwise the n <= max_splits
# minimising rounds(n)/n, the fewest within 5 % of the best; clamp to
# [1, min(ideal, 2 x SMs)] with ideal = cdiv(max_seq_len, min_work_per_split).

def test_num_kv_splits_single_round(lib):
    # 2 requests x cdiv(4*128, 64) = 8 row blocks -> 16 programs; 152 slots -> 9
    assert pkv.num_kv_splits(8192, 2, 4, 128, 152, 64, 1.0, 64, 8) == 9
    # capped by ideal = cdiv(100, 64) = 2
    assert pkv.num_kv_splits(100, 2, 4, 128, 152, 64, 1.0, 64, 8) == 2


def test_num_kv_splits_multi_round():
    # 32 requests x 8 row blocks = 256 programs on 152 slots:
    # n=1: 2 rounds -> 2.0; n=2: cdiv(512,152)=4 -> 2.0; n=3: 6/3=2.0;
    # n=4: cdiv(1024,152)=7 -> 1.75; n=5: 9/5=1.8; n=6: 11/6=1.83;
    # n=7: 12/7=1.714; n=8: 14/8=1.75  -> best 1.714; within 5%: <= 1.8 -> n=4
    assert pkv.num_kv_splits(8192, 32, 4, 128, 152, 64, 1.0, 64, 8) == 4
    # max_splits 1 -> 1
    assert pkv.num_kv_splits(8192, 32, 4, 128, 152, 64, 1.0, 64, 1) == 1


def test_num_kv_splits_clamps():
    # 2 x SMs cap: one program per split, 1000 slots, ideal large -> min(1000, 2*4)
    assert pkv.num_kv_splits(1 << 20, 1, 1, 1, 4, 64, 250.0, 1, 8) == 8
    assert pkv.num_kv_splits(0, 0, 1, 8, 152, 64, 1.0, 64, 8) == 1
    with pytest.raises(pkv.PkvError):
        pkv.num_kv_splits(8192, 2, 4, 128, 0, 64, 1.0, 64, 8)


def test_mla_entry_point_is_exported(lib):
    assert hasattr(lib, "pkv_mla_verify_attn")


# ------------------------------------------------------------- KV append --
def _append_args(B=2, Hkv=2, P=16, nb=64, maxb=8):
    return dict(k=_t([B, Hkv, 128], pkv.DTYPE_BF16), v=_t([B, Hkv, 128], pkv.DTYPE_BF16, ptr=0x20000),
                kv=_t([nb, Hkv, P, 256], pkv.DTYPE_BF16, ptr=0x30000),
                bt=_t([B, maxb], pkv.DTYPE_I32), sl=_t([B], pkv.DTYPE_I32))


def _append(lib, a, P=16):
    r = ctypes.byref
    return lib.pkv_gqa_kv_append(r(a["k"]), r(a["v"]), r(a["kv"]), r(a["bt"]), r(a["sl"]), P, None)


@pytest.mark.parametrize("mutate,P,code", [
    (lambda a: a.update(k=_t([2, 2, 64], pkv.DTYPE_BF16)), 16, -2),               # head dim
    (lambda a: a.update(v=_t([2, 3, 128], pkv.DTYPE_BF16)), 16, -1),              # v shape
    (lambda a: a.update(kv=_t([64, 4, 16, 256], pkv.DTYPE_BF16)), 16, -1),        # Hkv
    (lambda a: None, 8, -2),                                                       # page size
    (lambda a: None, 32, -1),                                                      # P != shape[2]
    (lambda a: a.update(k=_t([2, 2, 128], pkv.DTYPE_BF16, ptr=0x10004)), 16, -3),  # alignment
    (lambda a: a.update(sl=_t([3], pkv.DTYPE_I32)), 16, -1),                      # batch
    (lambda a: a.update(k=_t([2, 2, 128], pkv.DTYPE_F32)), 16, -1),               # dtype
])
def test_gqa_append_validation_rejects_before_any_cuda_call(lib, mutate, P, code):
    a = _append_args()
    mutate(a)
    assert _append(lib, a, P) == code
    assert pkv.last_error()


def test_gqa_append_empty_batch_is_a_no_op(lib):
    assert _append(lib, _append_args(B=0)) == 0


def test_mla_append_validation(lib):
    r = ctypes.byref
    lat = _t([8, 576], pkv.DTYPE_BF16)
    cache = _t([32, 16, 1, 576], pkv.DTYPE_FP8, ptr=0x40000)
    bt, sl = _t([4, 8], pkv.DTYPE_I32), _t([4], pkv.DTYPE_I32)
    ks = _t([], pkv.DTYPE_F32, ptr=0x50000)
    assert lib.pkv_mla_kv_append(r(lat), r(cache), r(bt), r(sl), 3, 16, r(ks), None) == -1  # 8 % 3
    assert lib.pkv_mla_kv_append(r(lat), r(cache), r(bt), r(sl), 2, 64, r(ks), None) == -2  # page
    bad = _t([8, 512], pkv.DTYPE_BF16)
    assert lib.pkv_mla_kv_append(r(bad), r(cache), r(bt), r(sl), 2, 16, r(ks), None) == -2  # Lk
    ks2 = _t([2], pkv.DTYPE_F32, ptr=0x50000)
    assert lib.pkv_mla_kv_append(r(lat), r(cache), r(bt), r(sl), 2, 16, r(ks2), None) == -1
    empty = _t([0, 576], pkv.DTYPE_BF16)
    bt0, sl0 = _t([0, 8], pkv.DTYPE_I32), _t([0], pkv.DTYPE_I32)
    assert lib.pkv_mla_kv_append(r(empty), r(cache), r(bt0), r(sl0), 2, 16, None, None) == 0


# --------------------------------------------------- native-FP8 MLA path --
def _nat_args(R=4, P=16):
    return dict(
        q8=_t([R, 128, 576], pkv.DTYPE_FP8), qs=_t([R, 128], pkv.DTYPE_F32, ptr=0x30000),
        c=_t([64, P, 1, 576], pkv.DTYPE_FP8), bt=_t([R, 8], pkv.DTYPE_I32),
        sl=_t([R], pkv.DTYPE_I32), out=_t([R, 128, 512], pkv.DTYPE_BF16, ptr=0x20000),
        lse=_t([R, 128], pkv.DTYPE_F32, ptr=0x40000))


def _nat_call(lib, a, qlen=1, P=16):
    r = ctypes.byref
    return lib.pkv_mla_verify_attn_fp8_native(r(a["q8"]), r(a["qs"]), r(a["c"]), r(a["bt"]),
                                              r(a["sl"]), None, qlen, 0.07, P, None,
                                              r(a["out"]), r(a["lse"]), 0, None)


@pytest.mark.parametrize("mutate,code", [
    (lambda a: a.update(c=_t([64, 16, 1, 576], pkv.DTYPE_BF16)), -2),          # bf16 cache
    (lambda a: a.update(q8=_t([4, 128, 576], pkv.DTYPE_BF16)), -1),            # q8 dtype
    (lambda a: a.update(q8=_t([4, 128, 576], pkv.DTYPE_FP8, ptr=0x10008)), -3),  # misaligned
    (lambda a: a.update(q8=_t([4, 128, 576], pkv.DTYPE_FP8, [73736, 576, 1])), -3),  # row stride
    (lambda a: a.update(qs=_t([4, 64], pkv.DTYPE_F32)), -1),                   # scale shape
    (lambda a: a.update(q8=_t([4, 64, 576], pkv.DTYPE_FP8),
                        qs=_t([4, 64], pkv.DTYPE_F32)), -2),                   # 64 heads
])
def test_native_validation_rejects_before_any_cuda_call(lib, mutate, code):
    a = _nat_args()
    mutate(a)
    assert _nat_call(lib, a) == code
    assert pkv.last_error()


def test_native_empty_batch_is_a_no_op(lib):
    assert _nat_call(lib, _nat_args(R=0)) == 0


@pytest.mark.parametrize("mutate,code", [
    (lambda a: a.update(q=_t([4, 128, 512], pkv.DTYPE_BF16)), -2),             # Lk 512
    (lambda a: a.update(q8=_t([4, 128, 576], pkv.DTYPE_FP8, [73728, 577, 1])), -3),
    (lambda a: a.update(q8=_t([4, 128, 576], pkv.DTYPE_FP8, ptr=0x10004)), -3),
    (lambda a: a.update(qs=_t([4, 128], pkv.DTYPE_BF16)), -1),
    (lambda a: a.update(q=_t([4, 128, 576], pkv.DTYPE_BF16, ptr=0x10002)), -3),
])
def test_quantize_validation_rejects_before_any_cuda_call(lib, mutate, code):
    a = dict(q=_t([4, 128, 576], pkv.DTYPE_BF16), q8=_t([4, 128, 576], pkv.DTYPE_FP8, ptr=0x50000),
             qs=_t([4, 128], pkv.DTYPE_F32, ptr=0x60000))
    mutate(a)
    r = ctypes.byref
    assert lib.pkv_mla_quantize_q(r(a["q"]), r(a["q8"]), r(a["qs"]), None) == code
    assert pkv.last_error()


# ------------------------------------------- overlapping outputs, any path --
def test_mla_outputs_overlapping_inputs_are_rejected(lib):
    def args():
        return dict(q8=_t([4, 128, 576], pkv.DTYPE_FP8, ptr=PTR["q"]),
                    qs=_t([4, 128], pkv.DTYPE_F32, ptr=PTR["sinks"]),
                    c=_t([64, 16, 1, 576], pkv.DTYPE_FP8, ptr=PTR["kv"]),
                    bt=_t([4, 8], pkv.DTYPE_I32, ptr=PTR["bt"]),
                    sl=_t([4], pkv.DTYPE_I32, ptr=PTR["sl"]),
                    out=_t([4, 128, 512], pkv.DTYPE_BF16, ptr=PTR["out"]),
                    lse=_t([4, 128], pkv.DTYPE_F32, ptr=PTR["lse"]))
    for name, ptr in (("out", PTR["q"] + 4096), ("out", PTR["kv"]), ("lse", PTR["out"] + 512),
                      ("lse", PTR["sinks"])):
        a = args()
        t = a[name]
        a[name] = _t([t.shape[i] for i in range(t.ndim)], t.dtype, ptr=ptr)
        assert _nat_call(lib, a) == -1, name
        assert "overlaps" in pkv.last_error()


def test_append_and_quantize_outputs_overlapping_inputs_are_rejected(lib):
    a = dict(k=_t([2, 2, 128], pkv.DTYPE_BF16, ptr=PTR["q"]),
             v=_t([2, 2, 128], pkv.DTYPE_BF16, ptr=PTR["out"]),
             kv=_t([64, 2, 16, 256], pkv.DTYPE_BF16, ptr=PTR["kv"]),
             bt=_t([2, 8], pkv.DTYPE_I32, ptr=PTR["bt"]), sl=_t([2], pkv.DTYPE_I32, ptr=PTR["sl"]))
    a["v"] = _t([2, 2, 128], pkv.DTYPE_BF16, ptr=PTR["kv"] + 8192)  # v inside the cache
    assert _append(lib, a) == -1 and "overlaps" in pkv.last_error()
    r = ctypes.byref
    q = _t([4, 128, 576], pkv.DTYPE_BF16, ptr=PTR["q"])
    q8 = _t([4, 128, 576], pkv.DTYPE_FP8, ptr=PTR["q"] + 65536)  # inside q
    qs = _t([4, 128], pkv.DTYPE_F32, ptr=PTR["lse"])
    assert lib.pkv_mla_quantize_q(r(q), r(q8), r(qs), None) == -1
    assert "overlaps" in pkv.last_error()


def test_block_table_width_times_page_size_must_fit_31_bits(lib):
    r = ctypes.byref
    lat = _t([8, 576], pkv.DTYPE_BF16, ptr=PTR["q"])
    cache = _t([32, 16, 1, 576], pkv.DTYPE_BF16, ptr=PTR["kv"])
    sl = _t([4], pkv.DTYPE_I32, ptr=PTR["sl"])
    wide = _t([4, 1 << 27], pkv.DTYPE_I32, ptr=PTR["bt"])  # 2^27 x 16 = 2^31
    assert lib.pkv_mla_kv_append(r(lat), r(cache), r(wide), r(sl), 2, 16, None, None) == -1
    assert "2^31" in pkv.last_error()
