"""Pins of the oracle's e4m3 query quantisation and of its quantised-query MLA
verify (the native-FP8 MLA path) against values fixed independently of it."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_30_gb300 import workloads as W

pytestmark = pytest.mark.filterwarnings("ignore")

LIB = None  # the oracle library under test (a mutant in test_oracle_mutants)


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


def bf16(a):
    return torch.tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


def test_quantize_scale_is_absmax_over_448_in_fp32():
    q = torch.randn(5, 3, 576, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    codes, scales = oracle.mla_quantize_q(q, lib=LIB)
    amax = q.float().abs().amax(dim=-1).numpy().astype(np.float32)
    np.testing.assert_array_equal(scales, amax / np.float32(448.0))


def test_quantize_absmax_element_is_448():
    q = torch.randn(4, 2, 576, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    codes, _ = oracle.mla_quantize_q(q, lib=LIB)
    qf = q.float().numpy()
    for r in range(4):
        for h in range(2):
            d = int(np.argmax(np.abs(qf[r, h])))
            assert oracle.e4m3_to_f64(int(codes[r, h, d])) == 448.0 * np.sign(qf[r, h, d])


def test_quantize_zero_row_and_single_value():
    q = np.zeros((1, 2, 576), dtype=np.float32)
    q[0, 1, 17] = -3.0
    codes, scales = oracle.mla_quantize_q(bf16(q), lib=LIB)
    assert scales[0, 0] == 1.0 and not codes[0, 0].any()
    assert scales[0, 1] == np.float32(3.0) / np.float32(448.0)
    assert oracle.e4m3_to_f64(int(codes[0, 1, 17])) == -448.0
    assert not np.delete(codes[0, 1], 17).any()


def test_quantize_matches_torch_float8_conversion_below_the_max():
    """Every element but the row maximum against PyTorch's own float8_e4m3fn
    rounding of the same fp32 quotient (round to nearest even)."""
    q = torch.randn(6, 4, 576, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    codes, scales = oracle.mla_quantize_q(q, lib=LIB)
    x = (q.float() / torch.from_numpy(scales)[..., None]).float()
    mask = x.abs() < 440.0
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert mask.sum() > 10000
    np.testing.assert_array_equal(codes[mask.numpy()], ref[mask.numpy()])


def test_quantize_error_within_half_a_step():
    """|code value x scale - q| <= 2^-4 |q| (normal range) or 2^-10 scale
    (subnormal range): half the e4m3 spacing."""
    q = torch.randn(3, 5, 576, generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    codes, scales = oracle.mla_quantize_q(q, lib=LIB)
    deq = np.vectorize(lambda c: oracle.e4m3_to_f64(int(c)))(codes) * scales[..., None]
    qf = q.double().numpy()
    bound = np.maximum(np.abs(qf) * 2.0 ** -4, scales[..., None] * 2.0 ** -10)
    assert np.all(np.abs(deq - qf) <= bound * (1 + 1e-12))


@pytest.mark.parametrize("shift", [0, 3])
def test_verify_q8_equals_verify_for_exactly_representable_queries(shift):
    """A query whose elements are e4m3 values times 2^-shift, with absmax
    448 x 2^-shift, quantises to scale 2^-shift and the very same codes: the
    quantised-query oracle then equals the bf16-query oracle bit for bit."""
    rng = np.random.default_rng(5 + shift)
    prob = W.mla_problem(9, B=3, qlen=2, H=128, page_size=16, lengths="const", Lmin=1,
                         Lmax=300, seq_lens=np.array([300, 17, 64], np.int32), fp8=True,
                         k_scale=0.05, has_real=False)
    grid = np.array([oracle.e4m3_to_f64(c) for c in range(0x7F) if c not in (0x7F,)])
    grid = grid[np.isfinite(grid)]
    vals = rng.choice(np.concatenate([grid, -grid]), size=prob.q.shape)
    vals[..., 5] = 448.0
    q = bf16(vals * 2.0 ** -shift)
    assert np.array_equal(q.float().numpy(), (vals * 2.0 ** -shift).astype(np.float32))
    codes, scales = oracle.mla_quantize_q(q, lib=LIB)
    assert np.all(scales == np.float32(2.0 ** -shift))
    ref_out, ref_lse = oracle.mla_verify(q, prob.latent_cache, prob.block_table, prob.seq_lens,
                                         None, prob.qlen, prob.scale, 16, prob.k_scale, lib=LIB)
    out, lse = oracle.mla_verify_q8(codes, scales, prob.latent_cache, prob.block_table,
                                    prob.seq_lens, None, prob.qlen, prob.scale, 16, prob.k_scale,
                                    lib=LIB)
    np.testing.assert_array_equal(out, ref_out)
    np.testing.assert_array_equal(lse, ref_lse)
