"""GPU parity of the MLA causal-verify kernel (tcgen05) against the fp64 oracle,
through the C ABI (pkv_mla_verify_attn via the ctypes binding)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_30_gb300 as pkv
from paged_kv_cache_30_gb300 import workloads as W
from tests.gpu_helpers import TOL_LSE, TOL_OUT, TOL_OUT_FP8, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    pkv.load_library()
    pkv.init(0)


def run_mla(prob, cap=None, dev=None):
    d = dev or dict(q=prob.q.cuda(), c=prob.latent_cache.cuda(), bt=prob.block_table.cuda(),
                    sl=prob.seq_lens.cuda(),
                    rl=None if prob.real_seq_lens is None else prob.real_seq_lens.cuda())
    R, H, _ = prob.q.shape
    out = torch.full((R, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((R, H), float("nan"), device="cuda")
    ks = None
    if prob.k_scale is not None:
        ks = torch.tensor(prob.k_scale, dtype=torch.float32, device="cuda")
    pkv.mla_verify_attn(d["q"], d["c"], d["bt"], d["sl"], d["rl"], prob.qlen, prob.scale,
                        prob.page_size, ks, out, lse,
                        prob.num_kv_splits if cap is None else cap)
    torch.cuda.synchronize()
    assert pkv.check_errors(0) == 0
    return out.float().cpu().numpy(), lse.cpu().numpy()


def oracle_mla(prob, rows=None):
    return oracle.mla_verify(prob.q, prob.latent_cache, prob.block_table, prob.seq_lens,
                             prob.real_seq_lens, prob.qlen, prob.scale, prob.page_size,
                             prob.k_scale, rows=rows)


def check(prob, cap=None, rows=None, what=""):
    out, lse = run_mla(prob, cap)
    ref_out, ref_lse = oracle_mla(prob, rows)
    R, H, _ = prob.q.shape
    tol = TOL_OUT_FP8 if prob.k_scale is not None else TOL_OUT
    if rows is None:
        return compare(out, lse, ref_out.reshape(R, H, 512), ref_lse.reshape(R, H), tol_out=tol,
                       what=what)
    return compare(out.reshape(-1, 512)[rows], lse.reshape(-1)[rows], ref_out, ref_lse,
                   tol_out=tol, what=what)


def mla_case(seed, L, qlen, P=16, real=None, Lmax=None, has_real=True, cap=0, poison=False):
    L = np.asarray(L, dtype=np.int32)
    prob = W.mla_problem(seed, B=len(L), qlen=qlen, H=128, page_size=P, lengths="const",
                         Lmin=1, Lmax=int(Lmax or max(int(L.max()), 1)), seq_lens=L,
                         has_real=has_real, num_kv_splits=cap)
    if real is not None:
        prob.real_seq_lens = torch.tensor(real, dtype=torch.int32)
    if poison:
        bt = prob.block_table.numpy()
        used = np.zeros(prob.latent_cache.shape[0], dtype=bool)
        used[bt[bt >= 0]] = True
        prob.latent_cache[torch.from_numpy(~used)] = float("nan")
        for b, l in enumerate(L):
            if l % P:
                prob.latent_cache[int(bt[b, (l - 1) // P]), l % P:] = float("nan")
    return prob


@pytest.mark.parametrize("seed,L,qlen,P,real,cap", [
    (0, [1, 31, 32, 33], 1, 16, None, 0),
    (1, [100, 1000], 4, 16, [97, 1000], 0),
    (2, [2500, 40, 5], 2, 32, [2500, 38, 0], 2),
    (3, [4097, 1500], 4, 16, None, 1),
    (4, [3000, 3000], 3, 16, [2999, 10], 3),
    (5, [70, 64, 63], 4, 32, None, 16),
    (6, [5000, 9, 700], 6, 16, [4998, 0, 700], 0),     # three token pairs, one request empty
    (7, [2049, 8000], 8, 32, [2049, 7993], 4),         # four token pairs, page 32
])
def test_mla_small_cases(seed, L, qlen, P, real, cap):
    prob = mla_case(seed, L, qlen, P, real=real, cap=cap)
    check(prob, what=f"mla case {seed}")


def test_mla_empty_rows_and_tiny_lengths():
    # lim = max(min(L - qlen + 1 + t, L_real), 0) is 0 for several rows here
    prob = mla_case(6, [2, 0, 1, 3], 4, 16, real=[2, 0, 0, 3])
    out, lse = run_mla(prob)
    ref_out, ref_lse = oracle_mla(prob)
    compare(out, lse, ref_out.reshape(out.shape), ref_lse.reshape(lse.shape), what="tiny")


def test_mla_poisoned_unattended_slots_stay_finite():
    prob = mla_case(7, [37, 200, 1025], 4, 16, real=[35, 200, 1024], poison=True)
    check(prob, what="mla poison")


def test_mla_degenerate_warmup_inputs():
    """All block-table entries point at page 0 and L = qlen (the verify page's
    warm-up runs every launch variant on such inputs)."""
    for qlen in (1, 2, 4):
        prob = mla_case(8, [qlen] * 3, qlen, 16, has_real=False)
        prob.block_table.zero_()
        for cap in (1, 2):
            check(prob, cap, what=f"warmup qlen {qlen} cap {cap}")


# Between two split counts of one MLA call.  Measured on GB300 (this test's
# problem and the B=32 qlen-4 workload, caps 1, 2, 5, 8, 16 against cap 1):
# outputs below 0.25 in magnitude differ by at most 1.95e-3: each split rounds
# P to bf16 against its own reference max, the same noise the GQA kernel's
# absolute 2e-3 bound covers.  Larger outputs (rows with few keys) add the
# final rounding: two fp32 results that differ by that noise round to bf16
# values up to one ulp further apart (worst seen: 3.9e-3 at |out| = 0.48,
# where an ulp is 2^-9, and 7.8e-3 at |out| = 1.08, where it is 2^-7).  lse
# differs by at most 9.5e-7.  Bound: every element within 2e-3 plus one bf16
# ulp of the larger magnitude; lse within 1e-5.
MLA_INV_ABS = 2e-3
MLA_INV_LSE = 1e-5


def check_split_invariance(outs, what):
    o1, l1 = outs[0]
    o1 = o1.astype(np.float64)
    for i, (out, lse) in enumerate(outs[1:], 1):
        out = out.astype(np.float64)
        mag = np.maximum(np.maximum(np.abs(out), np.abs(o1)), 2.0 ** -100)
        ulp = 2.0 ** (np.floor(np.log2(mag)) - 7)
        excess = np.abs(out - o1) - (MLA_INV_ABS + ulp)
        assert np.all(excess <= 0), \
            f"{what} #{i}: out beyond 2e-3 + 1 bf16 ulp from cap 1 (by {excess.max():.3g})"
        fin = np.isfinite(l1)
        assert np.array_equal(fin, np.isfinite(lse))
        d_lse = float(np.max(np.abs(lse[fin] - l1[fin]))) if fin.any() else 0.0
        assert d_lse <= MLA_INV_LSE, f"{what} #{i}: lse differs by {d_lse:.3g} from cap 1"


def test_mla_split_count_invariance():
    prob = mla_case(9, [6000, 3333], 4, 16, real=[5998, 3333])
    caps = (1, 2, 5, 8, 16)
    outs = [run_mla(prob, cap) for cap in caps]
    ref_out, ref_lse = oracle_mla(prob)
    for cap, (out, lse) in zip(caps, outs):
        compare(out, lse, ref_out.reshape(out.shape), ref_lse.reshape(lse.shape), what="inv")
    check_split_invariance(outs, "mla inv")


def test_mla_repeated_calls_are_bitwise_identical():
    prob = mla_case(10, [5000, 2000, 700], 4, 16)
    d = dict(q=prob.q.cuda(), c=prob.latent_cache.cuda(), bt=prob.block_table.cuda(),
             sl=prob.seq_lens.cuda(), rl=prob.real_seq_lens.cuda())
    first = run_mla(prob, dev=d)
    for _ in range(20):
        again = run_mla(prob, dev=d)
        assert np.array_equal(first[0], again[0]) and np.array_equal(first[1], again[1])
    assert pkv.check_counters(0) == 0


def test_mla_verify_b32_full_size_every_row():
    """B=32, qlen=4, H=128, L ~ U[512, 8192], L_real = L - U[0,3]: every
    (row, head) against the oracle in the benchmark's launch configuration
    (cap 8), and at caps 1 and 2 (split-count invariance)."""
    prob = W.mla_verify(0)
    R, H, _ = prob.q.shape
    ref_out, ref_lse = oracle_mla(prob)
    outs = []
    for cap in (1, 2, 8):
        out, lse = run_mla(prob, cap)
        compare(out, lse, ref_out.reshape(R, H, 512), ref_lse.reshape(R, H),
                what=f"mla config b32 q4 cap {cap}")
        outs.append((out, lse))
    check_split_invariance(outs, "mla b32 q4")


def test_mla_pair_split_size_both_branches():
    """The planning kernel splits CTA-pair launches at 6144 keys when every
    CTA pair still gets a unit at that size, else at 4096.  Eight requests of
    9000 keys with qlen 2 (32 units at 6144 keys: fewer than the CTA pairs of
    a GB300, so three 4096-key splits each) and forty of 6200..9000 keys (160
    units: two 6144-key splits each): every (row, head) against the oracle,
    unsplit (cap 1), at the library's split cap and at cap 8, and the caps
    agree within the split-invariance bound."""
    rng = np.random.default_rng(31)
    for seed, L in ((31, np.full(8, 9000)),
                    (32, rng.integers(6200, 9001, size=40))):
        L = L.astype(np.int32)
        real = np.maximum(L - rng.integers(0, 2, size=len(L)), 0).astype(np.int32)
        prob = mla_case(seed, L, 2, 16, real=real)
        ref_out, ref_lse = oracle_mla(prob)
        R, H, _ = prob.q.shape
        outs = []
        for cap in (1, 0, 8):
            out, lse = run_mla(prob, cap)
            compare(out, lse, ref_out.reshape(R, H, 512), ref_lse.reshape(R, H),
                    what=f"mla pair split B={len(L)} cap {cap}")
            outs.append((out, lse))
        check_split_invariance(outs, f"mla pair split B={len(L)}")
    assert pkv.check_counters(0) == 0


@pytest.mark.parametrize("seed,L,qlen,real,k_scale,cap,P", [
    (11, [64, 1, 1500], 1, None, 0.05, 0, 16),
    (12, [3000, 33], 4, [2998, 33], 0.05, 2, 16),
    (13, [700, 2049], 2, None, 0.125, 16, 16),
    (14, [2000, 65, 31], 3, [1999, 65, 31], 0.05, 0, 32),   # 32-token pages: two boxes a page
    (15, [5000, 1], 1, None, 0.02, 4, 32),
])
def test_mla_fp8_small_cases(seed, L, qlen, real, k_scale, cap, P):
    L = np.asarray(L, dtype=np.int32)
    prob = W.mla_problem(seed, B=len(L), qlen=qlen, H=128, page_size=P, lengths="const",
                         Lmin=1, Lmax=int(L.max()), seq_lens=L, fp8=True, k_scale=k_scale,
                         has_real=real is not None, num_kv_splits=cap)
    if real is not None:
        prob.real_seq_lens = torch.tensor(real, dtype=torch.int32)
    check(prob, what=f"fp8 case {seed}")


def test_mla_fp8_b128_full_size_every_row():
    """B=128, qlen=1, H=128, e4m3 latent cache holding N(0,1)/k_scale, k_scale
    0.05, log-uniform L in [1, 32768], cap 16: every (row, head)."""
    check(W.mla_fp8(0), what="mla fp8 b128")


def test_mla_request_order_paths():
    """Longest-first scheduling: 300 requests with many equal lengths (ranks
    broken by request index) and 520 requests (beyond the ranking limit, plain
    request order) -- every row against the oracle."""
    rng = np.random.default_rng(14)
    for B, seed in ((300, 14), (520, 15)):
        L = rng.choice([1, 17, 33, 40], size=B).astype(np.int32)
        prob = mla_case(seed, L, 1, 16, has_real=False, cap=2)
        check(prob, what=f"mla order B={B}")


def test_mla_plan_beyond_sort_limit():
    """8200 requests, above the planning kernel's 8192-request sort: units in
    request order with a fixed CTA slot per (request, split), most slots idle;
    six requests long enough for two splits.  A larger workspace holds the
    16400 x 2 partial slots.  Sampled rows (and rows of every long request)
    against the oracle."""
    rng = np.random.default_rng(21)
    B = 8200
    L = rng.choice([1, 17, 33, 40], size=B).astype(np.int32)
    long_idx = rng.choice(B, size=6, replace=False)
    L[long_idx] = [4100, 5000, 4097, 4500, 6000, 4200]
    prob = W.mla_problem(21, B=B, qlen=1, H=128, page_size=16, lengths="const", Lmin=1,
                         Lmax=int(L.max()), seq_lens=L, has_real=False, num_kv_splits=2)
    rows = np.concatenate([rng.choice(B * 128, size=512, replace=False),
                           (long_idx[:, None] * 128 + np.arange(0, 128, 16)).ravel()])
    pkv.shutdown()
    try:
        pkv.init(0, 6 << 30)
        check(prob, rows=rows, what="mla plan B=8200")
        assert pkv.check_counters(0) == 0
    finally:
        pkv.shutdown()
        pkv.init(0)
