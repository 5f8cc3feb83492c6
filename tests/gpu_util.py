"""Shared helpers of the GPU tests: conversions to the oracle's fp64 and tolerances.

Tolerances (from the stated parity bar):
  LSE                        |delta| <= 1e-3
  scores                     relative <= 2e-3; for log-domain scores (ln s, the surrogate's
                             predicted ln s+) that is |delta| <= 2e-3 in the log
  masks                      identical except keys whose oracle score lies within 1e-3
                             (relative on s, absolute on ln s) of tau or of the k-th value
  compaction                 bit-exact given the mask
"""
import numpy as np
import pytest
import torch

import oracle as O

LSE_ATOL = 1e-3
LOG_SCORE_ATOL = 2e-3
SCORE_RTOL = 2e-3
MASK_BAND = 1e-3


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def f64(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> exact float64 numpy array."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return O.bf16_bits_to_f64(t.view(torch.int16).numpy().view(np.uint16))
    return t.double().numpy()


def cuda(x: dict) -> dict:
    out = {}
    for k, v in x.items():
        out[k] = [t.cuda() for t in v] if isinstance(v, list) else v.cuda()
    return out


def assert_close_abs(got, want, atol, what):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    both_inf = np.isinf(got) & np.isinf(want) & (np.sign(got) == np.sign(want))
    err = np.where(both_inf, 0.0, np.abs(got - want))
    bad = ~(err <= atol)
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} beyond {atol}; max err {np.nanmax(err)}"


def assert_close_rel(got, want, rtol, what, atol=0.0):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    err = np.abs(got - want)
    bad = ~(err <= rtol * np.abs(want) + atol)
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} beyond rel {rtol}; "
                           f"max rel {np.nanmax(err / np.maximum(np.abs(want), 1e-300))}")


def assert_masks_match_near(mask_gpu, mask_ref, score_ref, pivots, band, what, log_domain):
    """Masks equal except where the oracle score is within `band` of a pivot (tau or the
    k-th value of that row).  pivots: array broadcastable to score_ref[..., :1]."""
    mask_gpu = np.asarray(mask_gpu).astype(bool)
    mask_ref = np.asarray(mask_ref).astype(bool)
    diff = mask_gpu != mask_ref
    if not diff.any():
        return
    piv = np.asarray(pivots, dtype=np.float64)[..., None]
    if log_domain:
        near = np.abs(score_ref - piv) <= band
    else:
        near = np.abs(score_ref - piv) <= band * np.abs(piv)
    assert not (diff & ~near).any(), f"{what}: {int((diff & ~near).sum())} mask differences away from the pivot"


def kth_value(score_ref, k, w):
    """Value of the k-th best candidate (outside the window) of each row, oracle order."""
    T = score_ref.shape[-1]
    flat = score_ref.reshape(-1, T)
    n = T - min(w, T)
    kk = min(k, n)
    out = np.full(flat.shape[0], np.nan)
    for r in range(flat.shape[0]):
        if 0 < kk:
            out[r] = flat[r, O.topk_order(flat[r, :n])[kk - 1]]
    return out.reshape(score_ref.shape[:-1])
