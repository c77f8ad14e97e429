"""GPU parity of the GQA paged decode kernel against the fp64 oracle, through
the C ABI (pkv_paged_decode_attn via the ctypes binding)."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_30_gb300 as pkv
from paged_kv_cache_30_gb300 import workloads as W
from tests.gpu_helpers import TOL_LSE, TOL_OUT, compare, dev, run_gqa

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
# Between two split counts of the same call: bf16 outputs within 2e-3, lse
# within 1e-4 (fp32 accumulation order only; each lane's running sum of the
# softmax denominator is compensated, so a single split of 131072 keys stays
# as accurate as many short ones).
LSE_INVARIANCE = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    pkv.load_library()
    pkv.init(0)


def oracle_gqa(prob, rows=None):
    return oracle.gqa_decode(prob.q, prob.kv_cache, prob.block_table, prob.seq_lens,
                             prob.sinks, prob.window, prob.scale, prob.page_size, rows=rows)


def check(prob, cap=None, what=""):
    out, lse = run_gqa(prob, cap)
    ref_out, ref_lse = oracle_gqa(prob)
    B, Hq, D = prob.q.shape
    return compare(out, lse, ref_out.reshape(B, Hq, D), ref_lse.reshape(B, Hq), what=what)


# ------------------------------------------------ the pages' worked example --

def test_block_table_worked_example_gpu():
    g = json.load(open(os.path.join(HERE, "golden", "block_table_example.json")))
    P, Hq, Hkv, D = g["page_size"], 8, 1, 128
    bt = np.array(g["block_table"], dtype=np.int32)
    L = np.array(g["seq_lens"], dtype=np.int32)
    kv = torch.full((g["num_pages"], Hkv, P, 2 * D), float("nan"))
    for b in range(len(L)):
        for j in range(L[b]):
            page, slot = int(bt[b, j // P]), j % P
            kv[page, :, slot, :D] = 0.0
            kv[page, :, slot, D:] = (32 * page + slot) / 256.0
    prob = W.GQAProblem(q=W.normal((3, Hq, D), 5), kv_cache=kv.to(torch.bfloat16),
                        block_table=torch.from_numpy(bt), seq_lens=torch.from_numpy(L),
                        sinks=None, window=0, scale=1 / math.sqrt(D), page_size=P)
    for cap in (1, 2, 0):
        out, lse = run_gqa(prob, cap)
        for b, e in enumerate(g["expected"]):
            n, d = map(int, e["out"].split("/"))
            exact = n / d
            # the GPU sums exact bf16 values in fp32 and rounds once to bf16
            assert np.all(np.abs(out[b] - exact) <= exact * 2.0 ** -8), (cap, b)
            assert np.max(np.abs(lse[b] - math.log(float(e["lse"][3:-1])))) <= 1e-5


# ----------------------------------------------------------- tiny workload --

@pytest.mark.parametrize("seed", range(5))
def test_tiny_gqa_config(seed):
    check(W.tiny_gqa(seed), what=f"tiny seed {seed}")


@pytest.mark.parametrize("seed,B,Hkv,P,Lmin,Lmax,sinks,window,cap", [
    (0, 3, 1, 16, 1, 700, True, 0, 0),
    (1, 5, 2, 16, 1, 1500, False, 0, 3),
    (2, 4, 3, 32, 1, 2100, True, 0, 0),
    (3, 6, 1, 32, 1, 999, True, 128, 0),
    (4, 7, 2, 16, 100, 3000, True, 37, 5),
    (5, 3, 4, 16, 16, 16, True, 0, 1),
    (6, 9, 1, 16, 1, 40, True, 0, 64),
    (7, 2, 2, 32, 1000, 5000, True, 1, 0),
    (8, 8, 1, 32, 31, 33, False, 32, 2),
    (9, 5, 2, 16, 1, 2000, True, 0, 1),      # cap 1: one item per (request, kv head)
    (10, 6, 1, 16, 1, 3000, True, 241, 0),   # widest window whose items never split at P 16
    (11, 6, 1, 16, 1, 3000, True, 242, 0),   # one token wider: the scanning prologue
])
@pytest.mark.parametrize("wide", [False, True])
def test_random_cases(seed, B, Hkv, P, Lmin, Lmax, sinks, window, cap, wide):
    """wide=False: block tables as wide as the longest request, so small
    launches whose requests may split take the cluster mode (splits merged
    through distributed shared memory); wide=True: the same problem with the
    tables padded to 1024 pages, which keeps the persistent kernel (queue,
    workspace partials, arrival counters)."""
    prob = W.gqa_problem(seed, B, 8 * Hkv, Hkv, P, "uniform", Lmin, Lmax, sinks=sinks,
                         window=window, num_kv_splits=cap, max_blocks=1024 if wide else None)
    check(prob, what=f"case {seed} wide={wide}")


def test_edge_lengths():
    """Empty rows, one key, exact page multiples, one past a page, window 1."""
    L = np.array([0, 1, 16, 17, 32, 33, 15, 0, 2, 48, 300, 257, 256, 513], dtype=np.int32)
    for window in (0, 1, 16, 17, 100):
        for P in (16, 32):
            for maxb in (None, 1024):  # cluster mode / persistent kernel
                prob = W.gqa_problem(11, len(L), 16, 2, P, "const", 1, 513, seq_lens=L,
                                     sinks=True, window=window, max_blocks=maxb)
                for cap in (1, 3, 0):
                    check(prob, cap, what=f"edge P={P} W={window} cap={cap} maxb={maxb}")


def test_nan_poisoned_unattended_slots_stay_finite():
    for P, window in ((16, 0), (32, 0), (16, 23), (32, 50)):
        prob = W.gqa_problem(12, 6, 16, 2, P, "uniform", 1, 600, sinks=True, window=window,
                             poison_unused=True)
        check(prob, what=f"poison P={P} W={window}")


def test_no_sinks_no_lse():
    prob = W.gqa_problem(13, 4, 8, 1, 16, "uniform", 1, 500)
    out, lse = run_gqa(prob, lse=False)
    ref_out, _ = oracle_gqa(prob)
    assert lse is None
    assert np.max(np.abs(out.reshape(ref_out.shape) - ref_out)) <= TOL_OUT


def test_strided_views():
    """q/out with padded batch rows and a cache whose kv heads are padded."""
    prob = W.gqa_problem(14, 4, 16, 2, 16, "uniform", 1, 400, sinks=True)
    B, Hq, D = prob.q.shape
    qbig = torch.zeros((B, Hq + 3, D), dtype=torch.bfloat16, device="cuda")
    qbig[:, :Hq] = prob.q.cuda()
    q = qbig[:, :Hq]
    nb, Hkv, P, D2 = prob.kv_cache.shape
    kvbig = torch.zeros((nb, Hkv + 1, P, D2), dtype=torch.bfloat16, device="cuda")
    kvbig[:, :Hkv] = prob.kv_cache.cuda()
    kv = kvbig[:, :Hkv]
    outbig = torch.zeros((B, Hq + 8, D), dtype=torch.bfloat16, device="cuda")
    out = outbig[:, 8:]
    lse = torch.empty((Hq, B), device="cuda").t()
    pkv.paged_decode_attn(q, kv, prob.block_table.cuda(), prob.seq_lens.cuda(),
                          prob.sinks.cuda(), 0, prob.scale, 16, 0, out, lse)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle_gqa(prob)
    compare(out.float().cpu().numpy(), lse.cpu().numpy(), ref_out.reshape(B, Hq, D),
            ref_lse.reshape(B, Hq), what="strided")
    assert torch.all(outbig[:, :8] == 0)


# ------------------------------------------------------------- invariants --

def test_split_count_invariance_and_counters_reset():
    prob = W.gqa_problem(15, 4, 32, 4, 32, "uniform", 2000, 9000, sinks=True)
    ref_out, ref_lse = oracle_gqa(prob)
    outs = []
    for cap in (1, 2, 8, 32, 132, 0):
        out, lse = run_gqa(prob, cap)
        compare(out, lse, ref_out.reshape(out.shape), ref_lse.reshape(lse.shape),
                what=f"cap {cap}")
        outs.append((out, lse))
    for out, lse in outs[1:]:
        assert np.max(np.abs(out - outs[0][0])) <= 2e-3
        assert np.max(np.abs(lse - outs[0][1])) <= LSE_INVARIANCE
    assert pkv.check_counters(0) == 0


def test_physical_page_permutation_is_bitwise_invariant():
    prob = W.gqa_problem(16, 5, 16, 2, 16, "uniform", 1, 3000, sinks=True)
    out1, lse1 = run_gqa(prob)
    nb = prob.kv_cache.shape[0]
    perm = torch.from_numpy(np.random.default_rng(5).permutation(nb))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(nb)
    bt2 = prob.block_table.clone()
    m = bt2 >= 0
    bt2[m] = inv[bt2[m].long()].int()
    prob2 = W.GQAProblem(q=prob.q, kv_cache=prob.kv_cache[perm].contiguous(), block_table=bt2,
                         seq_lens=prob.seq_lens, sinks=prob.sinks, window=0, scale=prob.scale,
                         page_size=16)
    out2, lse2 = run_gqa(prob2)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)


def test_repeated_calls_are_bitwise_identical():
    """The split schedule and merge order are fixed by seq_lens, so repeated
    calls must agree to the bit.  (Regression: a TMA refill of a ring stage
    overtaking the consumers' ldmatrix reads showed up as ~1 % of calls
    differing in one (request, kv head).)"""
    prob = W.gqa_problem(20, 16, 64, 8, 16, "uniform", 1000, 8000, sinks=True)
    q, kv, bt, sl, sk = (dev(prob.q), dev(prob.kv_cache), dev(prob.block_table),
                         dev(prob.seq_lens), dev(prob.sinks))
    outs = [torch.empty_like(q) for _ in range(200)]
    lses = [torch.empty(q.shape[:2], device="cuda") for _ in range(200)]
    for o, l in zip(outs, lses):
        pkv.paged_decode_attn(q, kv, bt, sl, sk, 0, prob.scale, 16, 0, o, l)
    torch.cuda.synchronize()
    differ = sum(int(not (torch.equal(o, outs[0]) and torch.equal(l, lses[0])))
                 for o, l in zip(outs, lses))
    assert differ == 0, f"{differ} of 200 calls differ"


def test_many_calls_leave_counters_at_zero():
    prob = W.gqa_problem(17, 8, 16, 2, 16, "uniform", 1, 4000, sinks=True)
    d = dict(q=dev(prob.q), kv=dev(prob.kv_cache), bt=dev(prob.block_table),
             sl=dev(prob.seq_lens), sinks=dev(prob.sinks))
    out = torch.empty_like(d["q"])
    for i in range(300):
        pkv.paged_decode_attn(d["q"], d["kv"], d["bt"], d["sl"], d["sinks"], 0, prob.scale, 16,
                              (0, 1, 4, 16)[i % 4], out, None)
    torch.cuda.synchronize()
    assert pkv.check_counters(0) == 0
    ref_out, _ = oracle_gqa(prob)
    assert np.max(np.abs(out.float().cpu().numpy().reshape(ref_out.shape) - ref_out)) <= TOL_OUT


@pytest.mark.parametrize("maxb", [200, 1024])  # cluster mode / persistent kernel
def test_cuda_graph_replay_with_new_lengths_and_tables(maxb):
    """The launch shape depends only on the batch: a captured call replays
    correctly after seq_lens and block_table change on the device."""
    pa = W.gqa_problem(18, 6, 16, 2, 16, "uniform", 1, 2000, sinks=True, max_blocks=maxb,
                       pool_pages=1200)
    pb = W.gqa_problem(19, 6, 16, 2, 16, "uniform", 1, 3000, sinks=True, max_blocks=maxb,
                       pool_pages=1200)
    pb.q = pa.q
    pb.sinks = pa.sinks
    pb.kv_cache = pa.kv_cache
    q, kv, sinks = dev(pa.q), dev(pa.kv_cache), dev(pa.sinks)
    bt, sl = dev(pa.block_table), dev(pa.seq_lens)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], device="cuda")
    s = torch.cuda.Stream()
    pkv.paged_decode_attn(q, kv, bt, sl, sinks, 0, pa.scale, 16, 0, out, lse, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pkv.paged_decode_attn(q, kv, bt, sl, sinks, 0, pa.scale, 16, 0, out, lse, stream=s)
    for prob in (pa, pb, pa):
        bt.copy_(prob.block_table.cuda())
        sl.copy_(prob.seq_lens.cuda())
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        ref_out, ref_lse = oracle_gqa(prob)
        compare(out.float().cpu().numpy(), lse.cpu().numpy(), ref_out.reshape(out.shape),
                ref_lse.reshape(lse.shape), what="graph replay")
    assert pkv.check_counters(0) == 0


def test_calls_on_two_streams_are_ordered():
    prob = W.gqa_problem(20, 16, 64, 8, 16, "uniform", 1000, 8000, sinks=True)
    q, kv, bt, sl, sk = (dev(prob.q), dev(prob.kv_cache), dev(prob.block_table),
                         dev(prob.seq_lens), dev(prob.sinks))
    outs = [torch.empty_like(q) for _ in range(4)]
    streams = [torch.cuda.Stream() for _ in range(2)]
    torch.cuda.synchronize()
    for i, o in enumerate(outs):
        pkv.paged_decode_attn(q, kv, bt, sl, sk, 0, prob.scale, 16, 0, o, None,
                              stream=streams[i % 2])
    torch.cuda.synchronize()
    ref_out, _ = oracle_gqa(prob)
    for o in outs:
        assert np.max(np.abs(o.float().cpu().numpy().reshape(ref_out.shape) - ref_out)) <= TOL_OUT
    assert pkv.check_counters(0) == 0


# --------------------------------------------------------- input errors --

@pytest.mark.parametrize("L", [100, 600])  # persistent kernel / cluster mode (3 splits)
def test_bad_block_table_entry_is_flagged_not_faulted(L):
    prob = W.gqa_problem(21, 3, 8, 1, 16, "const", L, L)
    bt = prob.block_table.clone()
    nb = prob.kv_cache.shape[0]
    bt[1, 2] = nb + 5          # past the end of the cache
    bt[2, 0] = -1              # unassigned entry inside the attended range
    bt[0, L // 16 - 1] = nb    # the last page of a later split
    q, kv, sl = dev(prob.q), dev(prob.kv_cache), dev(prob.seq_lens)
    out = torch.empty_like(q)
    pkv.paged_decode_attn(q, kv, bt.cuda(), sl, None, 0, prob.scale, 16, 0, out, None)
    with pytest.raises(pkv.PkvError) as ei:
        pkv.check_errors(0)
    assert ei.value.code == -7
    # the device stays usable and the next call is exact again
    check(prob, what="after bad table")


def test_bounded_wait_gives_up_and_reports_without_fault():
    """Failure detection without a GPU fault: one CTA waits on an mbarrier that
    nothing arrives on, through the kernels' bounded wait.  After about a
    second the wait gives up, bit 4 of the device error word is raised and
    pkv_check_errors reports it; the context stays usable (the next decode
    matches the oracle)."""
    import ctypes
    lib = pkv.load_library()
    flags = ctypes.c_int32(0)
    lib.pkv_check_errors(0, ctypes.byref(flags))  # start from a clear word
    pkv.selftest_wait_timeout(0)
    torch.cuda.synchronize()
    with pytest.raises(pkv.PkvError) as ei:
        pkv.check_errors(0)
    assert ei.value.code == -6 and "0x4" in str(ei.value)
    assert pkv.check_errors(0) == 0  # read and cleared
    check(W.gqa_problem(22, 3, 16, 2, 16, "uniform", 1, 900, sinks=True),
          what="after a timed-out wait")


@pytest.mark.parametrize("window, cap, maxb", [(0, 0, 4), (128, 0, 4), (0, 1, 4), (0, 0, 40),
                                               (0, 3, 40)])
def test_seq_len_beyond_block_table_is_flagged(window, cap, maxb):
    # (128, 0) and (0, 1): no request can split, so the kernel skips the
    # scanning prologue and checks the lengths as it decodes each item;
    # maxb 40: the cluster mode checks them as it decodes its split
    prob = W.gqa_problem(22, 2, 8, 1, 16, "const", 64, 64, max_blocks=maxb)
    sl = prob.seq_lens.clone()
    sl[0] = 1000
    out = torch.empty_like(dev(prob.q))
    pkv.paged_decode_attn(dev(prob.q), dev(prob.kv_cache), dev(prob.block_table), sl.cuda(),
                          None, window, prob.scale, 16, cap, out, None)
    with pytest.raises(pkv.PkvError) as ei:
        pkv.check_errors(0)
    assert ei.value.code == -7


def test_capture_before_workspace_is_refused_message():
    """Covered on the host: the first call allocates; an init during capture
    is refused (the workspace already exists here, so init is a no-op)."""
    pkv.init(0)  # idempotent
    assert pkv.check_counters(0) == 0


# ----------------------------------------------- full-size workloads ------

@pytest.mark.parametrize("window", [0, 128])
def test_flint_b64_full_size(window):
    """B=64, Hq=64, Hkv=8, page 16, log-uniform lengths up to 32768, sinks:
    every output row against the oracle, in the launch configuration the
    benchmark times (library-chosen split cap)."""
    prob = W.flint_gqa(0, window=window)
    check(prob, what=f"flint W={window}")


# The split counts the long-context stress sweeps (1, 8, 32, 132), plus the
# library's own choice (0).
LONG_CAPS = (0, 1, 8, 32, 132)


@pytest.mark.parametrize("B", [1, 8])
def test_long_context_split_sweep_every_row(B):
    """131072 keys per request, Hq=64, Hkv=8, page 32, pages scattered over a
    40960-page pool: every output row and lse at every split cap against the
    oracle, and every cap against cap 1 (split-count invariance)."""
    prob = W.long_context(0, B=B)
    ref_out, ref_lse = oracle_gqa(prob)
    ref_out = ref_out.reshape(B, 64, 128)
    ref_lse = ref_lse.reshape(B, 64)
    d = dict(q=dev(prob.q), kv=dev(prob.kv_cache), bt=dev(prob.block_table),
             sl=dev(prob.seq_lens), sinks=dev(prob.sinks))
    del prob.kv_cache
    outs = {}
    for cap in LONG_CAPS:
        out, lse = run_gqa(prob, cap, dev_tensors=d)
        compare(out, lse, ref_out, ref_lse, what=f"long B={B} cap {cap}")
        outs[cap] = (out, lse)
    o1, l1 = outs[1]
    for cap, (out, lse) in outs.items():
        # split-count invariance: fp32 accumulation order only
        assert np.max(np.abs(out - o1)) <= 2e-3, f"B={B} cap {cap}: out vs cap 1"
        assert np.max(np.abs(lse - l1)) <= LSE_INVARIANCE, f"B={B} cap {cap}: lse vs cap 1"
    del d
    torch.cuda.empty_cache()


def test_inputs_outside_device_memory_are_rejected_before_launch():
    """The call's device is the device holding q: a q in host memory (pinned or
    pageable) is refused with PKV_ERR_INVALID_ARG and nothing is written."""
    import ctypes
    prob = W.tiny_gqa(0)
    d = dict(kv=dev(prob.kv_cache), bt=dev(prob.block_table), sl=dev(prob.seq_lens))
    out = torch.full((4, 8, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    lib = pkv.load_library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    D = pkv._desc
    for q in (prob.q.clone(), prob.q.pin_memory()):
        for entry in ("pkv_paged_decode_attn", "pkv_paged_decode_attn_noalloc"):
            rc = getattr(lib, entry)(D(q), D(d["kv"]), D(d["bt"]), D(d["sl"]), None, 0,
                                     float(prob.scale), 16, 4, D(out), None, stream)
            assert rc == -1 and "not device memory" in pkv.last_error(), entry
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all()
