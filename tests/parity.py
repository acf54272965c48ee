"""Shared helpers of the GPU parity tests: moving seeded inputs to the device,
computing the oracle on the same values, and comparing within the tolerances
the grouped-query attention forward is held to:

  bf16 inputs, fp32 accumulation:  max |out - ref| <= 2e-2, mean |out - ref| <= 2e-3,
                                   max |lse - ref| <= 1e-3 on finite entries
  fp32 check mode:                 max |out - ref| <= 1e-5,  max |lse - ref| <= 1e-5

Entries whose reference lse is -inf (no admissible key) must be -inf on the
GPU too, with an all-zero output row.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

BF16_MAX, BF16_MEAN, BF16_LSE = 2e-2, 2e-3, 1e-3
FP32_MAX, FP32_LSE = 1e-5, 1e-5


def tol_for(dtype):
    if dtype == torch.bfloat16:
        return BF16_MAX, BF16_MEAN, BF16_LSE
    return FP32_MAX, FP32_MAX, FP32_LSE


def to_dev(d, device="cuda"):
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def compare(got, ref, dtype, what="out", max_tol=None, mean_tol=None):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "%s has non-finite values" % what
    tmax, tmean, _ = tol_for(dtype)
    tmax = tmax if max_tol is None else max_tol
    tmean = tmean if mean_tol is None else mean_tol
    err = np.abs(got - ref)
    emax, emean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
    where = np.unravel_index(int(err.argmax()), err.shape) if err.size else ()
    msg = "%s: max-abs %.3g (at %s) mean-abs %.3g rel-l2 %.3g" % (what, emax, where, emean, rel)
    assert emax <= tmax and emean <= tmean, msg
    return emax, emean, rel


def compare_lse(got, ref, dtype):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    neg = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), neg), "lse -inf pattern differs"
    _, _, tl = tol_for(dtype)
    if (~neg).any():
        e = float(np.abs(got[~neg] - ref[~neg]).max())
        assert e <= tl, "lse max-abs %.3g > %.3g" % (e, tl)


def oracle_fwd(inp, scale, causal, rows=None):
    return oracle.attention(inp["q"], inp["k"], inp["v"], scale=scale, causal=causal,
                            seqlens_k=inp.get("seqlens_k"), rows=rows)


def gather_rows(out, lse, rows, Sq, Hq):
    """Pick (b,h,i) rows from out [B,Sq,Hq,D] and lse [B,Hq,Sq] (CPU float64 arrays)."""
    rows = np.asarray(rows)
    i = rows % Sq
    h = (rows // Sq) % Hq
    b = rows // (Sq * Hq)
    return out[b, i, h, :], lse[b, h, i]
