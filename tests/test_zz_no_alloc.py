"""The allocation-free GQA entry point (pkv_paged_decode_attn_noalloc), for
callers that cannot let a library allocate device memory: it must agree with
the allocating entry point, call after call, on the same inputs.

This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_30_gb300 as pkv
from paged_kv_cache_30_gb300 import workloads as W
from tests.gpu_helpers import TOL_LSE, TOL_OUT

pytestmark = pytest.mark.gpu


def _inputs(prob):
    return dict(q=prob.q.cuda(), kv=prob.kv_cache.cuda(), bt=prob.block_table.cuda(),
                sl=prob.seq_lens.cuda(), sinks=None if prob.sinks is None else prob.sinks.cuda())


def _run(entry, prob, d, cap):
    """One call through the C ABI; returns (out, lse) on the host."""
    lib = pkv.load_library()
    out = torch.full_like(d["q"], float("nan"))
    lse = torch.full(d["q"].shape[:2], float("nan"), device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    D = pkv._desc
    rc = getattr(lib, entry)(D(d["q"]), D(d["kv"]), D(d["bt"]), D(d["sl"]), D(d["sinks"]),
                             prob.window, float(prob.scale), prob.page_size, cap, D(out), D(lse),
                             stream)
    assert rc == 0, pkv.last_error()
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


def _agree(a, b):
    assert np.all(np.isfinite(a[0])) and np.all(np.isfinite(b[0]))
    assert np.max(np.abs(a[0] - b[0])) <= TOL_OUT
    fin = np.isfinite(b[1])
    assert np.array_equal(fin, np.isfinite(a[1]))
    assert np.max(np.abs(a[1][fin] - b[1][fin]), initial=0.0) <= TOL_LSE


def test_noalloc_matches_allocating_entry_point_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    pkv.load_library()
    cases = [
        # (problem, cap): two different calls back to back, so the second one
        # starts from whatever the first left in the shared scratch
        (W.gqa_problem(101, 16, 64, 8, 16, "loguniform", 1, 8000, sinks=True), 0),
        (W.gqa_problem(102, 9, 32, 4, 32, "uniform", 1, 6000, sinks=True, window=300), 7),
    ]
    inputs = [_inputs(p) for p, _ in cases]
    refs = [_run("pkv_paged_decode_attn", p, d, c) for (p, c), d in zip(cases, inputs)]
    free = []
    for rep in range(2):
        for (p, c), d, ref in zip(cases, inputs, refs):
            got = _run("pkv_paged_decode_attn_noalloc", p, d, c)
            _agree(got, ref)
        torch.cuda.synchronize()
        free.append(torch.cuda.mem_get_info()[0])
    # The first call loads the library module that holds the static scratch;
    # after that, calls take no device memory (the torch caching allocator
    # only serves this test's own output tensors, below 1 MiB).
    assert free[1] >= free[0] - (1 << 20)


def test_noalloc_rejects_calls_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    prob = W.gqa_problem(103, 64, 64, 8, 16, "uniform", 1, 200)  # 512 pairs
    d = _inputs(prob)
    out = torch.empty_like(d["q"])
    with pytest.raises(pkv.PkvError) as ei:
        # 512 pairs x 8 splits = 4096 partials > 2048
        pkv.paged_decode_attn_noalloc(d["q"], d["kv"], d["bt"], d["sl"], None, 0, prob.scale, 16,
                                      8, out, None)
    assert ei.value.code == -4 and "2048" in str(ei.value)
