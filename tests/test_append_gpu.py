"""GPU parity of the paged KV append (pkv_gqa_kv_append, pkv_mla_kv_append)
against the oracle: byte-exact, over the whole cache."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_30_gb300 as pkv
from paged_kv_cache_30_gb300 import workloads as W
from tests.gpu_helpers import TOL_LSE, TOL_OUT, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    pkv.load_library()
    pkv.init(0)


def _u(t):
    """Raw bits of a CPU or GPU tensor as a numpy array."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.numpy()


def _gqa_case(seed, L, Hkv, P, max_blocks=None):
    L = np.asarray(L, dtype=np.int32)
    prob = W.gqa_problem(seed, B=len(L), Hq=8 * Hkv, Hkv=Hkv, page_size=P, lengths="const",
                         Lmin=1, Lmax=max(int(L.max()), 1), seq_lens=L, max_blocks=max_blocks)
    k = W.normal((len(L), Hkv, 128), seed * 31 + 5)
    v = W.normal((len(L), Hkv, 128), seed * 31 + 6)
    return prob, k, v


@pytest.mark.parametrize("seed,L,Hkv,P", [
    (0, [1, 16, 17, 33, 0, 300], 2, 16),
    (1, [32, 31, 64, 65, 1000], 8, 32),
    (2, list(range(1, 70)), 1, 16),
])
def test_gqa_append_matches_oracle_bytewise(seed, L, Hkv, P):
    prob, k, v = _gqa_case(seed, L, Hkv, P)
    want, skipped = oracle.gqa_kv_append(k, v, prob.kv_cache, prob.block_table, prob.seq_lens, P)
    assert skipped == 0
    kv = prob.kv_cache.cuda()
    pkv.gqa_kv_append(k.cuda(), v.cuda(), kv, prob.block_table.cuda(), prob.seq_lens.cuda(), P)
    torch.cuda.synchronize()
    assert pkv.check_errors(0) == 0
    assert np.array_equal(_u(kv), want)


def test_gqa_append_bad_entries_are_flagged_and_not_written():
    prob, k, v = _gqa_case(3, [20, 40, 5], 2, 16, max_blocks=3)
    bt = prob.block_table.clone()
    bt[0, 1] = -1                              # position 19 -> logical page 1: unassigned
    sl = prob.seq_lens.clone()
    sl[1] = 3 * 16 + 5                         # beyond the table
    want, skipped = oracle.gqa_kv_append(k, v, prob.kv_cache, bt, sl, 16)
    assert skipped == 2
    kv = prob.kv_cache.cuda()
    pkv.gqa_kv_append(k.cuda(), v.cuda(), kv, bt.cuda(), sl.cuda(), 16)
    torch.cuda.synchronize()
    with pytest.raises(pkv.PkvError):
        pkv.check_errors(0)
    assert np.array_equal(_u(kv), want)


@pytest.mark.parametrize("fp8,qlen,P", [(False, 1, 16), (False, 4, 32), (True, 1, 16),
                                        (True, 4, 16), (True, 3, 32)])
def test_mla_append_matches_oracle_bytewise(fp8, qlen, P):
    L = np.array([4, 17, 33, 64, 2, 500], dtype=np.int32)
    prob = W.mla_problem(20 + qlen, B=len(L), qlen=qlen, H=128, page_size=P, lengths="const",
                         Lmin=1, Lmax=int(L.max()), seq_lens=L, fp8=fp8, k_scale=0.05,
                         has_real=False)
    lat = W.normal((len(L) * qlen, 576), 77 + qlen)
    ks = prob.k_scale if fp8 else None
    want, skipped = oracle.mla_kv_append(lat, prob.latent_cache, prob.block_table,
                                         prob.seq_lens, qlen, P, k_scale=ks)
    assert skipped == 0
    cache = prob.latent_cache.cuda()
    kst = torch.tensor(ks, dtype=torch.float32, device="cuda") if fp8 else None
    pkv.mla_kv_append(lat.cuda(), cache, prob.block_table.cuda(), prob.seq_lens.cuda(), qlen, P,
                      kst)
    torch.cuda.synchronize()
    assert pkv.check_errors(0) == 0
    assert np.array_equal(_u(cache), want)


def test_mla_fp8_append_rounds_ties_and_saturates():
    """Values at e4m3 midpoints (ties to even) and beyond 448 after the
    division by k_scale, against the oracle's encoder."""
    ks = 0.25
    codes = np.arange(0, 0x7E, dtype=np.int64)
    lo = np.array([oracle.e4m3_to_f64(int(c)) for c in codes])
    hi = np.array([oracle.e4m3_to_f64(int(c) + 1) for c in codes])
    vals = np.concatenate([(lo + hi) / 2, -(lo + hi) / 2, [500.0, -1000.0, 1e4]]) * ks
    vals = vals[np.abs(vals) < 3e38]
    x = torch.from_numpy(vals.astype(np.float32)).to(torch.bfloat16)
    n = (x.numel() + 575) // 576 * 576
    lat = torch.zeros(n, dtype=torch.bfloat16)
    lat[: x.numel()] = x
    lat = lat.view(-1, 576)
    R = lat.shape[0]
    bt = torch.arange(R, dtype=torch.int32).view(R, 1)
    sl = torch.ones(R, dtype=torch.int32)
    cache = torch.zeros((R, 16, 1, 576), dtype=torch.float8_e4m3fn)
    want, _ = oracle.mla_kv_append(lat, cache, bt, sl, 1, 16, k_scale=ks)
    c = cache.cuda()
    pkv.mla_kv_append(lat.cuda(), c, bt.cuda(), sl.cuda(), 1, 16,
                      torch.tensor(ks, dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    assert np.array_equal(_u(c), want)


def test_gqa_append_full_size_then_decode():
    """The Flint-shaped batch: append every request's current token into the
    full cache (only those rows change), then decode: equal to the oracle's
    decode of the oracle-appended cache on sampled rows."""
    prob = W.flint_gqa(0, 0)
    B, Hq = prob.q.shape[:2]
    Hkv = Hq // 8
    k = W.normal((B, Hkv, 128), 91)
    v = W.normal((B, Hkv, 128), 92)
    kv = prob.kv_cache.cuda()
    before = kv.clone()
    bt, sl = prob.block_table.cuda(), prob.seq_lens.cuda()
    pkv.gqa_kv_append(k.cuda(), v.cuda(), kv, bt, sl, prob.page_size)
    torch.cuda.synchronize()
    assert pkv.check_errors(0) == 0
    changed = (kv.view(torch.int16) != before.view(torch.int16)).any(dim=-1).nonzero().cpu()
    del before
    L = prob.seq_lens.numpy()
    expect = set()
    for b in range(B):
        if L[b] > 0:
            pos = int(L[b]) - 1
            blk = int(prob.block_table[b, pos // prob.page_size])
            expect |= {(blk, h, pos % prob.page_size) for h in range(Hkv)}
    assert {tuple(int(x) for x in r) for r in changed} <= expect
    rows_kv = kv[[e[0] for e in sorted(expect)], [e[1] for e in sorted(expect)],
                 [e[2] for e in sorted(expect)]].cpu()
    kk = {}
    for b in range(B):
        if L[b] > 0:
            pos = int(L[b]) - 1
            blk = int(prob.block_table[b, pos // prob.page_size])
            for h in range(Hkv):
                kk[(blk, h, pos % prob.page_size)] = torch.cat([k[b, h], v[b, h]])
    assert torch.equal(rows_kv.view(torch.int16),
                       torch.stack([kk[e] for e in sorted(expect)]).view(torch.int16))
    # decode on the appended cache vs the oracle on its own appended copy
    new_cache, _ = oracle.gqa_kv_append(k, v, prob.kv_cache, prob.block_table, prob.seq_lens,
                                        prob.page_size)
    out = torch.empty_like(prob.q, device="cuda")
    lse = torch.empty((B, Hq), device="cuda")
    pkv.paged_decode_attn(prob.q.cuda(), kv, bt, sl, prob.sinks.cuda(), 0, prob.scale,
                          prob.page_size, prob.num_kv_splits, out, lse)
    torch.cuda.synchronize()
    rows = np.random.default_rng(5).choice(B * Hq, size=256, replace=False)
    ref_out, ref_lse = oracle.gqa_decode(prob.q, torch.from_numpy(new_cache.view(np.int16)).view(
        torch.bfloat16), prob.block_table, prob.seq_lens, prob.sinks, 0, prob.scale,
        prob.page_size, rows=rows)
    compare(out.float().cpu().numpy().reshape(-1, 128)[rows], lse.cpu().numpy().reshape(-1)[rows],
            ref_out, ref_lse, tol_out=TOL_OUT, tol_lse=TOL_LSE, what="append then decode")
