"""Helpers shared by the GPU parity tests: upload a seeded problem, run the
CUDA library through its binding, compare with the oracle."""
import numpy as np
import torch

import paged_kv_cache_30_gb300 as pkv

# Tolerances (max abs error) stated for this path: bf16 outputs 2e-2, 5e-2
# with an FP8 cache, natural-log LSE 1e-3.
TOL_OUT = 2e-2
TOL_OUT_FP8 = 5e-2
TOL_LSE = 1e-3


def within_bf16_reorder(a, b, ulps=2.0, floor=1e-4):
    """True when two runs of one call that only accumulate in a different
    order agree: each element within `ulps` bf16 ulps of the larger magnitude
    (each side rounds once to bf16), or within `floor` absolute for values
    near zero, where fp32 cancellation (terms of size ~1) dominates."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    mag = np.maximum(np.maximum(np.abs(a), np.abs(b)), 2.0 ** -100)
    ulp = 2.0 ** (np.floor(np.log2(mag)) - 7)
    return bool(np.all(np.abs(a - b) <= np.maximum(ulps * ulp, floor)))


def dev(t):
    return None if t is None else t.to("cuda", non_blocking=False)


def run_gqa(prob, cap=None, lse=True, stream=None, dev_tensors=None):
    """Run pkv_paged_decode_attn on the problem; returns (out fp32 numpy, lse)."""
    d = dev_tensors or dict(q=dev(prob.q), kv=dev(prob.kv_cache), bt=dev(prob.block_table),
                            sl=dev(prob.seq_lens), sinks=dev(prob.sinks))
    out = torch.empty_like(d["q"])
    out.fill_(float("nan"))
    lse_t = torch.full((prob.q.shape[0], prob.q.shape[1]), float("nan"), device="cuda") \
        if lse else None
    pkv.paged_decode_attn(d["q"], d["kv"], d["bt"], d["sl"], d["sinks"], prob.window,
                          prob.scale, prob.page_size,
                          prob.num_kv_splits if cap is None else cap, out, lse_t, stream=stream)
    torch.cuda.synchronize()
    flags = pkv.check_errors(0)
    assert flags == 0, f"device error word {flags:#x}"
    return out.float().cpu().numpy(), (lse_t.cpu().numpy() if lse else None)


def compare(out, lse, ref_out, ref_lse, tol_out=TOL_OUT, tol_lse=TOL_LSE, what=""):
    out = np.asarray(out, dtype=np.float64).reshape(ref_out.shape)
    assert np.all(np.isfinite(out)), f"{what}: non-finite output"
    err = np.max(np.abs(out - ref_out)) if out.size else 0.0
    assert err <= tol_out, f"{what}: max |out - oracle| = {err:.3e} > {tol_out}"
    if lse is not None:
        lse = np.asarray(lse, dtype=np.float64).reshape(ref_lse.shape)
        fin = np.isfinite(ref_lse)
        assert np.array_equal(fin, np.isfinite(lse)), f"{what}: lse finiteness differs"
        assert np.all(np.isneginf(lse[~fin])), f"{what}: empty rows must have lse = -inf"
        if fin.any():
            e2 = np.max(np.abs(lse[fin] - ref_lse[fin]))
            assert e2 <= tol_lse, f"{what}: max |lse - oracle| = {e2:.3e} > {tol_lse}"
    return err
