"""The allocation-free GQA entry point (pkv_paged_decode_attn_noalloc).

It serves callers that cannot let a library allocate device memory: a serving
engine that has handed all of HBM to its own KV-cache pool, or a framework
whose memory manager must own every device buffer.  Its results must agree
with the allocating entry point and with the oracle, call after call, on the
same inputs, and its limits must hold exactly at the scratch array's edges.

This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_30_gb300 as pkv
from paged_kv_cache_30_gb300 import workloads as W
from tests.gpu_helpers import TOL_LSE, TOL_OUT, compare

pytestmark = pytest.mark.gpu

# The static scratch's limits (stated in include/pkv.h).
MAX_PAIRS = 4096
MAX_PARTIALS = 2048


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    pkv.load_library()


def _inputs(prob):
    return dict(q=prob.q.cuda(), kv=prob.kv_cache.cuda(), bt=prob.block_table.cuda(),
                sl=prob.seq_lens.cuda(), sinks=None if prob.sinks is None else prob.sinks.cuda())


def _call(entry, prob, d, cap, stream=None):
    """One call through the C ABI; returns (rc, out, lse) with out/lse on the host."""
    lib = pkv.load_library()
    out = torch.full_like(d["q"], float("nan"))
    lse = torch.full(d["q"].shape[:2], float("nan"), device="cuda")
    if stream is None:
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    D = pkv._desc
    rc = getattr(lib, entry)(D(d["q"]), D(d["kv"]), D(d["bt"]), D(d["sl"]), D(d["sinks"]),
                             prob.window, float(prob.scale), prob.page_size, cap, D(out), D(lse),
                             stream)
    torch.cuda.synchronize()
    return rc, out.float().cpu().numpy(), lse.cpu().numpy()


def _run(entry, prob, d, cap):
    rc, out, lse = _call(entry, prob, d, cap)
    assert rc == 0, pkv.last_error()
    assert pkv.check_errors(0) == 0
    return out, lse


def _agree(a, b):
    assert np.all(np.isfinite(a[0])) and np.all(np.isfinite(b[0]))
    assert np.max(np.abs(a[0] - b[0])) <= TOL_OUT
    fin = np.isfinite(b[1])
    assert np.array_equal(fin, np.isfinite(a[1]))
    assert np.max(np.abs(a[1][fin] - b[1][fin]), initial=0.0) <= TOL_LSE


def _oracle(prob):
    ro, rl = oracle.gqa_decode(prob.q, prob.kv_cache, prob.block_table, prob.seq_lens,
                               prob.sinks, prob.window, prob.scale, prob.page_size)
    B, Hq, D = prob.q.shape
    return ro.reshape(B, Hq, D), rl.reshape(B, Hq)


def test_noalloc_matches_allocating_entry_point_on_two_calls_in_a_row():
    cases = [
        # (problem, cap): two different calls back to back, so the second one
        # starts from whatever the first left in the shared scratch
        (W.gqa_problem(101, 16, 64, 8, 16, "loguniform", 1, 8000, sinks=True), 0),
        (W.gqa_problem(102, 9, 32, 4, 32, "uniform", 1, 6000, sinks=True, window=300), 7),
    ]
    inputs = [_inputs(p) for p, _ in cases]
    refs = [_run("pkv_paged_decode_attn", p, d, c) for (p, c), d in zip(cases, inputs)]
    oracles = [_oracle(p) for p, _ in cases]
    free = []
    for rep in range(2):
        for (p, c), d, ref, (ro, rl) in zip(cases, inputs, refs, oracles):
            got = _run("pkv_paged_decode_attn_noalloc", p, d, c)
            _agree(got, ref)
            compare(got[0], got[1], ro, rl, what=f"no-alloc seed {p.meta.get('seed', '')} #{rep}")
            if c != 0:
                # an explicit cap gives both entry points the same launch shape
                # (one host helper computes it), so the same bits
                assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])
        torch.cuda.synchronize()
        free.append(torch.cuda.mem_get_info()[0])
    # The first call loads the library module that holds the static scratch;
    # after that, calls take no device memory (the torch caching allocator
    # only serves this test's own output tensors, below 1 MiB).
    assert free[1] >= free[0] - (1 << 20)


@pytest.mark.parametrize("B,Hkv,cap", [
    (128, 8, 2),      # 1024 pairs x 2 splits = 2048 partials: the limit, splits allowed
    (512, 8, 0),      # 4096 pairs, library cap: 2048 / 4096 rounds to one split per pair
    (2048, 2, 1),     # 4096 pairs at cap 1: no partials needed
])
def test_noalloc_at_the_scratch_limits_matches_the_oracle(B, Hkv, cap):
    prob = W.gqa_problem(104, B, 8 * Hkv, Hkv, 16, "uniform", 1, 700, sinks=True)
    d = _inputs(prob)
    ro, rl = _oracle(prob)
    for _ in range(2):
        out, lse = _run("pkv_paged_decode_attn_noalloc", prob, d, cap)
        compare(out, lse, ro, rl, what=f"no-alloc limit B={B} Hkv={Hkv} cap={cap}")
    assert pkv.check_counters(0) == 0  # the allocating workspace is untouched


@pytest.mark.parametrize("B,Hkv,cap,what", [
    (683, 1, 3, "2048 split partials"),   # 683 pairs x 3 = 2049 partials
    (241, 17, 1, "4096"),                 # 4097 pairs
    (64, 8, 8, "2048 split partials"),    # 512 pairs x 8 = 4096 partials
])
def test_noalloc_rejects_calls_one_past_its_scratch(B, Hkv, cap, what):
    prob = W.gqa_problem(105, B, 8 * Hkv, Hkv, 16, "uniform", 1, 40)
    d = _inputs(prob)
    rc, out, _ = _call("pkv_paged_decode_attn_noalloc", prob, d, cap)
    assert rc == -4 and what in pkv.last_error()
    assert np.all(np.isnan(out))  # nothing was launched


def test_noalloc_device_errors_reach_check_errors():
    prob = W.gqa_problem(106, 3, 8, 1, 16, "const", 1, 100, sinks=True)
    prob.block_table[1, 2] = prob.kv_cache.shape[0] + 5  # a page outside the cache
    d = _inputs(prob)
    rc, out, _ = _call("pkv_paged_decode_attn_noalloc", prob, d, 0)
    assert rc == 0
    flags = ctypes.c_int32(0)
    lib = pkv.load_library()
    assert lib.pkv_check_errors(0, ctypes.byref(flags)) == -7  # PKV_ERR_BAD_BLOCK_TABLE
    assert flags.value & 1
    assert lib.pkv_check_errors(0, ctypes.byref(flags)) == 0 and flags.value == 0  # cleared
