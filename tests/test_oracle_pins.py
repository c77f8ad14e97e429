"""Pins for the fp64 CPU oracle: each test checks the oracle against something
other than itself -- values printed on the pages (the transformers block-table
example), library routines (torch's bf16 / float8 decoders, scipy's softmax and
logsumexp on dense inputs), closed forms and invariants of attention.

A wrong index, a dropped term, a wrong sign or a transposed operand in the
oracle fails at least one of these; ``test_oracle_mutants.py`` plants such
mistakes in copies of the oracle and checks that they do.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special as sps
import torch

import oracle
from paged_kv_cache_30_gb300 import workloads as W

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden")

# The oracle library under test: None = the built oracle.  The mutation tests
# point this at deliberately broken copies and expect these pins to fail.
LIB = None


def gqa(*args, **kw):
    return oracle.gqa_decode(*args, lib=LIB, **kw)


def mla(*args, **kw):
    return oracle.mla_verify(*args, lib=LIB, **kw)


# ---------------------------------------------------------------- decoders --

def test_bf16_decode_matches_torch_all_codes(oracle_lib):
    codes = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    ref = codes.view(torch.bfloat16).double().numpy()
    got = np.array([oracle_lib.pkv_oracle_bf16_to_f64(c & 0xFFFF) for c in range(1 << 16)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


def test_e4m3_decode_matches_torch_all_codes(oracle_lib):
    codes = torch.arange(0, 256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle_lib.pkv_oracle_e4m3_to_f64(c) for c in range(256)])
    nan = np.isnan(ref)
    assert nan.sum() == 2  # S.1111.111, both signs
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


# ------------------------------------------------- the pages' worked example --

def _frac(s):
    n, d = s.split("/")
    return int(n) / int(d)


def _ln(s):
    assert s.startswith("ln(") and s.endswith(")")
    return math.log(float(s[3:-1]))


def block_table_example(Hq=8, Hkv=1, D=128):
    """The transformers block-table example as a GQA problem (K = 0, V encodes
    page and slot, NaN everywhere that must not be read)."""
    g = json.load(open(os.path.join(GOLDEN, "block_table_example.json")))
    P, npages = g["page_size"], g["num_pages"]
    bt = np.array(g["block_table"], dtype=np.int32)
    L = np.array(g["seq_lens"], dtype=np.int32)
    kv = torch.full((npages, Hkv, P, 2 * D), float("nan"), dtype=torch.float32)
    for b in range(len(L)):
        for j in range(L[b]):
            page, slot = int(bt[b, j // P]), j % P
            kv[page, :, slot, :D] = 0.0
            kv[page, :, slot, D:] = (32 * page + slot) / 256.0
    q = W.normal((len(L), Hq, D), 5)
    prob = W.GQAProblem(q=q, kv_cache=kv.to(torch.bfloat16), block_table=torch.from_numpy(bt),
                        seq_lens=torch.from_numpy(L), sinks=None, window=0,
                        scale=1.0 / math.sqrt(D), page_size=P)
    exp_out = np.array([_frac(e["out"]) for e in g["expected"]])
    exp_lse = np.array([_ln(e["lse"]) for e in g["expected"]])
    return prob, exp_out, exp_lse


@pytest.mark.parametrize("Hq,Hkv", [(1, 1), (8, 1)])
def test_block_table_worked_example(Hq, Hkv):
    prob, exp_out, exp_lse = block_table_example(Hq, Hkv)
    out, lse = gqa(prob.q, prob.kv_cache, prob.block_table, prob.seq_lens,
                                 None, 0, prob.scale, prob.page_size)
    out = out.reshape(3, Hq, -1)
    lse = lse.reshape(3, Hq)
    assert np.all(np.isfinite(out))
    for b in range(3):
        assert np.max(np.abs(out[b] - exp_out[b])) <= 1e-12
        assert np.max(np.abs(lse[b] - exp_lse[b])) <= 1e-12


def test_block_table_example_unassigned_entry_is_an_error():
    """Reading a -1 entry is an input error, never a silent read."""
    prob, _, _ = block_table_example()
    L = prob.seq_lens.clone()
    L[0] = 33  # needs block_table[0][1] == -1
    with pytest.raises(oracle.OracleError):
        gqa(prob.q, prob.kv_cache, prob.block_table, L, None, 0,
                          prob.scale, prob.page_size)


# ------------------------------------------- dense attention via scipy ------

def dense_reference(prob, window=0):
    """softmax(scale * q K^T) V with scipy, on keys gathered densely by torch
    indexing; a sink is an extra key with logit `sink` and a zero value row."""
    q = prob.q.double().numpy()
    kv = prob.kv_cache.double().numpy()
    bt = prob.block_table.numpy()
    L = prob.seq_lens.numpy()
    B, Hq, D = q.shape
    Hkv, P = kv.shape[1], kv.shape[2]
    G = Hq // Hkv
    sc = float(np.float32(prob.scale))
    out = np.zeros((B, Hq, D))
    lse = np.full((B, Hq), -np.inf)
    for b in range(B):
        s = max(L[b] - window, 0) if window > 0 else 0
        pos = np.arange(s, L[b])
        if len(pos) == 0:
            continue
        pages, slots = bt[b, pos // P], pos % P
        for h in range(Hq):
            K = kv[pages, h // G, slots, :D]
            V = kv[pages, h // G, slots, D:]
            x = sc * (K @ q[b, h])
            lse[b, h] = sps.logsumexp(x)
            if prob.sinks is not None:
                xs = np.concatenate([x, [float(prob.sinks[h])]])
                out[b, h] = sps.softmax(xs)[:-1] @ V
            else:
                out[b, h] = sps.softmax(x) @ V
    return out, lse


def _tiny(seed, B, Hq, Hkv, P, Lmax, sinks=False, window=0, D=128, identity=True, Lmin=0):
    rng = np.random.default_rng(seed)
    L = rng.integers(Lmin, Lmax + 1, size=B).astype(np.int32)
    maxb = (Lmax + P - 1) // P + 1
    if identity:
        # contiguous cache: request b's logical page i is physical page b*maxb + i
        bt = (np.arange(B)[:, None] * maxb + np.arange(maxb)[None, :]).astype(np.int32)
        kv = W.normal((B * maxb, Hkv, P, 2 * D), seed + 100)
        prob = W.GQAProblem(q=W.normal((B, Hq, D), seed + 101), kv_cache=kv,
                            block_table=torch.from_numpy(bt), seq_lens=torch.from_numpy(L),
                            sinks=W.normal((Hq,), seed + 102, torch.float32) if sinks else None,
                            window=window, scale=1.0 / math.sqrt(D), page_size=P)
        return prob
    return W.gqa_problem(seed, B, Hq, Hkv, P, "uniform", Lmin, Lmax, D=D, sinks=sinks,
                         window=window, seq_lens=L, max_blocks=maxb)


@pytest.mark.parametrize("seed,B,Hq,Hkv,P,Lmax,sinks,window", [
    (0, 3, 1, 1, 16, 64, False, 0),
    (1, 3, 8, 1, 16, 64, True, 0),
    (2, 2, 16, 2, 32, 64, True, 0),
    (3, 3, 8, 1, 16, 64, False, 20),
    (4, 3, 8, 1, 4, 40, True, 7),
    (5, 2, 4, 4, 8, 33, True, 0),
])
def test_oracle_matches_dense_scipy(seed, B, Hq, Hkv, P, Lmax, sinks, window):
    prob = _tiny(seed, B, Hq, Hkv, P, Lmax, sinks, window)
    ref_out, ref_lse = dense_reference(prob, window)
    out, lse = gqa(prob.q, prob.kv_cache, prob.block_table, prob.seq_lens,
                                 prob.sinks, window, prob.scale, P)
    out = out.reshape(ref_out.shape)
    lse = lse.reshape(ref_lse.shape)
    assert np.max(np.abs(out - ref_out)) <= 1e-12
    fin = np.isfinite(ref_lse)
    assert np.array_equal(fin, np.isfinite(lse))
    assert np.max(np.abs(lse[fin] - ref_lse[fin]), initial=0.0) <= 1e-12


def test_oracle_random_block_table_matches_dense():
    prob = _tiny(7, 3, 8, 1, 16, 120, sinks=True, identity=False)
    ref_out, ref_lse = dense_reference(prob)
    out, lse = gqa(prob.q, prob.kv_cache, prob.block_table, prob.seq_lens,
                                 prob.sinks, 0, prob.scale, 16)
    assert np.max(np.abs(out.reshape(ref_out.shape) - ref_out)) <= 1e-12
    assert np.max(np.abs(lse.reshape(ref_lse.shape) - ref_lse)) <= 1e-12


# ------------------------------------------------------------- invariants --

def test_single_key_returns_v_exactly():
    prob = _tiny(11, 3, 8, 1, 16, 64)
    prob.seq_lens[:] = 1
    out, lse = gqa(prob.q, prob.kv_cache, prob.block_table, prob.seq_lens,
                                 None, 0, prob.scale, 16)
    out = out.reshape(3, 8, 128)
    for b in range(3):
        v0 = prob.kv_cache[int(prob.block_table[b, 0]), 0, 0, 128:].double().numpy()
        assert np.array_equal(out[b], np.broadcast_to(v0, (8, 128)))
    # single key: lse equals that key's scaled score
    s = np.array([float(np.float32(prob.scale)) *
                  (prob.q[b, h].double() @ prob.kv_cache[int(prob.block_table[b, 0]), 0, 0, :128]
                   .double()).item() for b in range(3) for h in range(8)])
    assert np.max(np.abs(lse - s)) <= 1e-12


def test_constant_v_returns_constant():
    prob = _tiny(12, 3, 8, 1, 16, 64, Lmin=1)
    prob.kv_cache[..., 128:] = 0.75
    out, _ = gqa(prob.q, prob.kv_cache, prob.block_table, prob.seq_lens,
                               None, 0, prob.scale, 16)
    assert np.max(np.abs(out - 0.75)) <= 1e-14


def test_empty_rows_write_zero_and_neg_inf_lse():
    prob = _tiny(13, 3, 8, 1, 16, 64, sinks=True)
    prob.seq_lens[1] = 0
    out, lse = gqa(prob.q, prob.kv_cache, prob.block_table, prob.seq_lens,
                                 prob.sinks, 0, prob.scale, 16)
    out = out.reshape(3, 8, 128)
    lse = lse.reshape(3, 8)
    assert np.all(out[1] == 0.0) and np.all(np.isneginf(lse[1]))
    assert np.all(np.isfinite(lse[[0, 2]][prob.seq_lens.numpy()[[0, 2]] > 0]))


def test_sink_limits():
    prob = _tiny(14, 3, 8, 1, 16, 64, Lmin=1)
    base, base_lse = gqa(prob.q, prob.kv_cache, prob.block_table, prob.seq_lens,
                                       None, 0, prob.scale, 16)
    ninf = torch.full((8,), float("-inf"))
    o1, l1 = gqa(prob.q, prob.kv_cache, prob.block_table, prob.seq_lens,
                               ninf, 0, prob.scale, 16)
    assert np.array_equal(o1, base) and np.array_equal(l1, base_lse)
    big = torch.full((8,), 80.0)
    o2, l2 = gqa(prob.q, prob.kv_cache, prob.block_table, prob.seq_lens,
                               big, 0, prob.scale, 16)
    assert np.max(np.abs(o2)) < 1e-20
    assert np.array_equal(l2, base_lse)  # the sink never enters lse
    # a sink equal to the key-only lse M + ln Z weighs as much as all keys
    # together, so it halves the output (up to the sink's fp32 rounding delta:
    # out = base / (1 + exp(delta)))
    lse0 = base_lse.reshape(3, 8)[0]
    sink = torch.tensor(lse0, dtype=torch.float32)
    o3, _ = gqa(prob.q[:1], prob.kv_cache, prob.block_table[:1],
                              prob.seq_lens[:1], sink, 0, prob.scale, 16)
    delta = sink.double().numpy() - lse0
    expect = base.reshape(3, 8, 128)[0] / (1.0 + np.exp(delta))[:, None]
    assert np.max(np.abs(o3.reshape(8, 128) - expect)) <= 1e-12


def test_physical_page_permutation_invariance():
    prob = _tiny(15, 3, 8, 1, 16, 120, sinks=True, identity=False)
    out, lse = gqa(prob.q, prob.kv_cache, prob.block_table, prob.seq_lens,
                                 prob.sinks, 0, prob.scale, 16)
    nb = prob.kv_cache.shape[0]
    perm = torch.from_numpy(np.random.default_rng(3).permutation(nb))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(nb)
    kv2 = prob.kv_cache[perm]             # new page i holds old page perm[i]
    bt2 = prob.block_table.clone()
    m = bt2 >= 0
    bt2[m] = inv[bt2[m].long()].int()
    out2, lse2 = gqa(prob.q, kv2, bt2, prob.seq_lens, prob.sinks, 0,
                                   prob.scale, 16)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_window_equals_full_attention_on_last_w_keys():
    prob = _tiny(16, 3, 8, 1, 16, 100, sinks=True, identity=True, Lmin=30)
    W_ = 17
    out_w, lse_w = gqa(prob.q, prob.kv_cache, prob.block_table, prob.seq_lens,
                                     prob.sinks, W_, prob.scale, 16)
    # shift every request so that its last W keys start at logical position 0
    P = 16
    for b in range(3):
        L = int(prob.seq_lens[b])
        kv_flat = []
        for j in range(L - W_, L):
            kv_flat.append(prob.kv_cache[int(prob.block_table[b, j // P]), :, j % P])
        sub = torch.stack(kv_flat)  # [W, Hkv, 2D]
        pages = (W_ + P - 1) // P
        kv_new = torch.zeros((pages, 1, P, 256), dtype=torch.bfloat16)
        for i in range(W_):
            kv_new[i // P, :, i % P] = sub[i]
        bt = torch.arange(pages, dtype=torch.int32)[None]
        o, l = gqa(prob.q[b:b + 1], kv_new, bt, torch.tensor([W_], dtype=torch.int32),
                                 prob.sinks, 0, prob.scale, P)
        assert np.array_equal(o, out_w.reshape(3, 8, 128)[b])
        assert np.array_equal(l, lse_w.reshape(3, 8)[b])


def test_head_grouping_uses_kv_head_h_div_group():
    """Give kv head g the constant value g+1 in V: query head h must read h // G + 1."""
    prob = _tiny(17, 2, 16, 2, 16, 40, Lmin=1)
    for g in range(2):
        prob.kv_cache[:, g, :, 128:] = float(g + 1)
    out, _ = gqa(prob.q, prob.kv_cache, prob.block_table, prob.seq_lens,
                               None, 0, prob.scale, 16)
    out = out.reshape(2, 16, 128)
    for h in range(16):
        assert np.max(np.abs(out[:, h] - float(h // 8 + 1))) <= 1e-14


# --------------------------------------------------------------------- MLA --

def mla_dense_reference(prob, lims):
    """Dense softmax over the first lims[r] keys of each verify row (scipy);
    V = the first Lv dims of the gathered latent K."""
    q = prob.q.double().numpy()
    c = prob.latent_cache
    ks = 1.0 if prob.k_scale is None else float(np.float32(prob.k_scale))
    cache = c.double().numpy() * ks
    P = prob.page_size
    cache = cache.reshape(-1, P, c.shape[-1])
    bt = prob.block_table.numpy()
    R, H, Lk = q.shape
    Lv = prob.Lv
    sc = float(np.float32(prob.scale))
    out = np.zeros((R, H, Lv))
    lse = np.full((R, H), -np.inf)
    for r in range(R):
        b = r // prob.qlen
        lim = lims[r]
        if lim == 0:
            continue
        pos = np.arange(lim)
        K = cache[bt[b, pos // P], pos % P]
        x = sc * (q[r] @ K.T)                     # [H, lim]
        lse[r] = sps.logsumexp(x, axis=1)
        out[r] = sps.softmax(x, axis=1) @ K[:, :Lv]
    return out, lse


def _mla_tiny(seed, B, qlen, H, P, L, real=None, fp8=False, Lk=576, Lv=512):
    prob = W.mla_problem(seed, B=B, qlen=qlen, H=H, page_size=P, lengths="const",
                         Lmin=1, Lmax=max(L) if len(L) else 1, Lk=Lk, Lv=Lv, fp8=fp8,
                         seq_lens=np.array(L, dtype=np.int32), has_real=real is not None)
    if real is not None:
        prob.real_seq_lens = torch.tensor(real, dtype=torch.int32)
    return prob


@pytest.mark.parametrize("fp8", [False, True])
def test_mla_qlen1_equals_dense_attention(fp8):
    prob = _mla_tiny(21, 3, 1, 16, 16, [1, 37, 64], fp8=fp8)
    ref_out, ref_lse = mla_dense_reference(prob, [1, 37, 64])
    out, lse = mla(prob.q, prob.latent_cache, prob.block_table, prob.seq_lens,
                                 None, 1, prob.scale, 16, prob.k_scale)
    assert np.max(np.abs(out.reshape(ref_out.shape) - ref_out)) <= 1e-12
    assert np.max(np.abs(lse.reshape(ref_lse.shape) - ref_lse)) <= 1e-12


@pytest.mark.parametrize("L,real,qlen,lims", [
    # row limit max(min(L - qlen + 1 + t, L_real), 0), values worked by hand
    ([10], None, 4, [7, 8, 9, 10]),
    ([10], [8], 4, [7, 8, 8, 8]),
    ([2], None, 4, [0, 0, 1, 2]),
    ([40, 5], [37, 0], 3, [37, 37, 37, 0, 0, 0]),
    ([33, 17], [33, 15], 2, [32, 33, 15, 15]),
])
def test_mla_verify_row_limits(L, real, qlen, lims):
    prob = _mla_tiny(22, len(L), qlen, 8, 16, L, real=real)
    ref_out, ref_lse = mla_dense_reference(prob, lims)
    out, lse = mla(prob.q, prob.latent_cache, prob.block_table, prob.seq_lens,
                                 prob.real_seq_lens, qlen, prob.scale, 16)
    out = out.reshape(ref_out.shape)
    lse = lse.reshape(ref_lse.shape)
    assert np.max(np.abs(out - ref_out)) <= 1e-12
    fin = np.isfinite(ref_lse)
    assert np.array_equal(fin, np.isfinite(lse))
    assert np.max(np.abs(lse[fin] - ref_lse[fin]), initial=0.0) <= 1e-12
    assert np.all(out[~fin] == 0.0)


def test_mla_v_is_the_leading_lv_dims_of_k():
    """A latent cache whose first Lv = 512 dims are a constant c returns c,
    whatever the remaining 64 dims hold: V is K[..., :Lv]."""
    prob = _mla_tiny(23, 2, 2, 8, 16, [20, 50])
    prob.latent_cache[..., :512] = 0.5
    out, _ = mla(prob.q, prob.latent_cache, prob.block_table, prob.seq_lens,
                               None, 2, prob.scale, 16)
    assert np.max(np.abs(out - 0.5)) <= 1e-14


def test_mla_fp8_k_scale_scales_v_and_scores():
    """Doubling k_scale doubles V and the logits: out(2s) with scale/2 == 2*out(s)."""
    prob = _mla_tiny(24, 2, 1, 8, 16, [19, 40], fp8=True)
    o1, l1 = mla(prob.q, prob.latent_cache, prob.block_table, prob.seq_lens,
                               None, 1, prob.scale, 16, 0.25)
    o2, l2 = mla(prob.q, prob.latent_cache, prob.block_table, prob.seq_lens,
                               None, 1, prob.scale / 2, 16, 0.5)
    assert np.max(np.abs(o2 - 2 * o1)) <= 1e-12
    assert np.max(np.abs(l2 - l1)) <= 1e-12
