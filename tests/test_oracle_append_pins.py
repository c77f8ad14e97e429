"""Pins of the oracle's paged KV append and e4m3 encoder (CPU only).

The append follows "Atencion paginada" (transformers), decode path: the new
token of a sequence with n cached tokens is written in place at logical
position n, i.e. page block_table[b][n / P], slot n % P; with the decode
kernel's seq_lens (Flint page: lengths including the current token) that is
position seq_lens - 1, and an MLA verify row t sits at seq_lens - qlen + t.
The e4m3 encoder follows the OCP float8 e4m3 "fn" definition (bias 7, 3
mantissa bits, subnormals, no infinity, largest finite 448): nearest value,
ties to even, saturating.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle

LIB = None  # swapped by the mutant tests
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_append_example.json")


def _lib():
    return LIB or oracle.load()


def _example():
    with open(GOLDEN) as f:
        g = json.load(f)
    bt = torch.tensor(g["block_table"], dtype=torch.int32)
    sl = torch.tensor(g["cache_seqlens"], dtype=torch.int32) + 1
    return g, bt, sl


def _bits(x):
    return torch.from_numpy(np.asarray(x, dtype=np.int16)).view(torch.bfloat16)


def test_gqa_append_worked_example():
    g, bt, sl = _example()
    P, nb, Hkv, D = g["page_size"], g["num_pages"], 2, 4
    rng = np.random.default_rng(0)
    cache = _bits(rng.integers(-2**15, 2**15, size=(nb, Hkv, P, 2 * D)))
    k = _bits(rng.integers(-2**15, 2**15, size=(3, Hkv, D)))
    v = _bits(rng.integers(-2**15, 2**15, size=(3, Hkv, D)))
    new, skipped = oracle.gqa_kv_append(k, v, cache, bt, sl, P, lib=_lib())
    assert skipped == 0
    old = cache.view(torch.int16).numpy().view(np.uint16)
    changed = np.argwhere(np.any(new != old, axis=-1))  # (block, head, slot)
    want = {(blk, h, slot) for blk, slot in g["expected_block_slot"] for h in range(Hkv)}
    assert {tuple(int(x) for x in c) for c in changed} <= want
    kb, vb = k.view(torch.int16).numpy().view(np.uint16), v.view(torch.int16).numpy().view(np.uint16)
    for b, (blk, slot) in enumerate(g["expected_block_slot"]):
        for h in range(Hkv):
            assert np.array_equal(new[blk, h, slot, :D], kb[b, h])
            assert np.array_equal(new[blk, h, slot, D:], vb[b, h])
    mask = np.ones(new.shape[:3], dtype=bool)
    for blk, slot in g["expected_block_slot"]:
        mask[blk, :, slot] = False
    assert np.array_equal(new[mask], old[mask])


@pytest.mark.parametrize("qlen", [1, 2])
def test_mla_append_worked_example(qlen):
    g, bt, sl = _example()
    P, nb, Lk = g["page_size"], g["num_pages"], 8
    rng = np.random.default_rng(1)
    cache = _bits(rng.integers(-2**15, 2**15, size=(nb, P, 1, Lk)))
    lat = _bits(rng.integers(-2**15, 2**15, size=(3 * qlen, Lk)))
    new, skipped = oracle.mla_kv_append(lat, cache, bt, sl, qlen, P, lib=_lib())
    assert skipped == 0
    # the new token of each sequence (row qlen-1) at the worked example's slot;
    # with qlen = 2 the row before it at the preceding position: sequence 1's
    # earlier row is position 31, the last slot of its first block 0
    where = {1: [[(2, 30)], [(1, 0)], [(6, 6)]],
             2: [[(2, 29), (2, 30)], [(0, 31), (1, 0)], [(6, 5), (6, 6)]]}[qlen]
    old = cache.view(torch.int16).numpy().view(np.uint16)
    lb = lat.view(torch.int16).numpy().view(np.uint16)
    mask = np.ones((nb, P), dtype=bool)
    for b in range(3):
        for t, (blk, slot) in enumerate(where[b]):
            assert np.array_equal(new[blk, slot, 0], lb[b * qlen + t])
            mask[blk, slot] = False
    assert np.array_equal(new[mask], old[mask])


def test_append_skips_rows_without_a_position_or_page():
    P, nb, Hkv, D = 16, 4, 1, 4
    bt = torch.tensor([[0, -1], [1, 2], [3, 1]], dtype=torch.int32)
    sl = torch.tensor([0, 17, 40], dtype=torch.int32)  # no token; page 1 -> block 2; beyond table
    cache = _bits(np.zeros((nb, Hkv, P, 2 * D), dtype=np.int16))
    k = _bits(np.full((3, Hkv, D), 0x3F80, dtype=np.int16))
    v = _bits(np.full((3, Hkv, D), 0x4000, dtype=np.int16))
    new, skipped = oracle.gqa_kv_append(k, v, cache, bt, sl, P, lib=_lib())
    assert skipped == 1
    assert np.count_nonzero(np.any(new != 0, axis=-1)) == 1
    assert np.all(new[2, 0, 0, :D] == 0x3F80) and np.all(new[2, 0, 0, D:] == 0x4000)
    bt2 = torch.tensor([[0, -1], [1, -1], [3, 1]], dtype=torch.int32)  # unassigned entry
    new2, skipped2 = oracle.gqa_kv_append(k, v, cache, bt2, sl, P, lib=_lib())
    assert skipped2 == 2 and not np.any(new2)


def _enc(x):
    return int(_lib().pkv_oracle_f32_to_e4m3(float(np.float32(x))))


def _dec(c):
    return oracle.e4m3_to_f64(c)


def test_e4m3_encode_round_trips_every_code():
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert _enc(_dec(c)) == c, hex(c)
    assert _enc(float("nan")) == 0x7F


def test_e4m3_encode_ties_to_even_and_saturates():
    pos = [c for c in range(0x7F)]  # 0 .. 448, increasing
    for c in pos[:-1]:
        lo, hi = _dec(c), _dec(c + 1)
        mid = (lo + hi) / 2
        even = c if c % 2 == 0 else c + 1
        assert _enc(mid) == even, hex(c)
        assert _enc(np.nextafter(np.float32(mid), np.float32(np.inf))) == c + 1
        assert _enc(np.nextafter(np.float32(mid), np.float32(-np.inf))) == c
        assert _enc(-mid) == even | 0x80
    assert _enc(448.0) == 0x7E and _enc(464.0) == 0x7E and _enc(1e30) == 0x7E
    assert _enc(-1e30) == 0xFE and _enc(float("inf")) == 0x7E
    assert _enc(2.0 ** -10) == 0x00 and _enc(3 * 2.0 ** -10) == 0x02
    assert _enc(-0.0) == 0x80 and _enc(0.0) == 0x00


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.normal(0, 1, 20000), rng.normal(0, 100, 20000),
                        rng.normal(0, 1e-2, 20000)]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([_enc(v) for v in x], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_mla_fp8_append_stores_e4m3_of_x_over_k_scale():
    P, nb, Lk, ks = 16, 2, 16, 0.05
    rng = np.random.default_rng(3)
    x = rng.normal(0, 1, size=(1, Lk)).astype(np.float32)
    x[0, 0] = 30.0  # 600 after division: saturates
    lat = torch.from_numpy(x).to(torch.bfloat16)
    cache = torch.zeros((nb, P, 1, Lk), dtype=torch.float8_e4m3fn)
    bt = torch.tensor([[1]], dtype=torch.int32)
    sl = torch.tensor([5], dtype=torch.int32)
    new, skipped = oracle.mla_kv_append(lat, cache, bt, sl, 1, P, k_scale=ks, lib=_lib())
    assert skipped == 0
    xb = lat.float().numpy()[0]
    want = [_enc(np.float32(v) / np.float32(ks)) for v in xb]
    assert list(new[1, 4, 0]) == want
    assert new[1, 4, 0, 0] == 0x7E
    assert np.count_nonzero(new) == np.count_nonzero(new[1, 4, 0])
