"""Tolerance checks shared by the GPU parity tests.

The bar (stated for this layer): with rms = sqrt(mean(o_ref^2)),
  max |o - o_ref| / rms <= 2e-2,   mean |o - o_ref| / rms <= 2e-3,
  ||S - S_ref||_F / ||S_ref||_F <= 1e-2.
"""
import numpy as np
import torch

MAX_REL, MEAN_REL, STATE_REL = 2e-2, 2e-3, 1e-2


def _np(x):
    if isinstance(x, torch.Tensor):
        return x.detach().float().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def output_errors(o, o_ref):
    o, o_ref = _np(o), _np(o_ref)
    rms = np.sqrt(np.mean(o_ref ** 2))
    d = np.abs(o - o_ref)
    return float(d.max() / rms), float(d.mean() / rms)


def state_error(s, s_ref):
    s, s_ref = _np(s), _np(s_ref)
    return float(np.linalg.norm((s - s_ref).ravel()) / np.linalg.norm(s_ref.ravel()))


def assert_output_close(o, o_ref, max_rel=MAX_REL, mean_rel=MEAN_REL, what="out"):
    mx, mn = output_errors(o, o_ref)
    assert np.isfinite(_np(o)).all(), f"{what}: non-finite values"
    assert mx <= max_rel and mn <= mean_rel, f"{what}: max/rms {mx:.3e}, mean/rms {mn:.3e}"
    return mx, mn


def assert_state_close(s, s_ref, rel=STATE_REL, what="state"):
    e = state_error(s, s_ref)
    assert np.isfinite(_np(s)).all(), f"{what}: non-finite values"
    assert e <= rel, f"{what}: ||dS||/||S|| = {e:.3e}"
    return e


def assert_bf16_output_close(o, o_ref, max_rel=MAX_REL, mean_rel=MEAN_REL, what="out"):
    """bf16 outputs: the bar above plus the storage rounding itself, i.e.
    |o - ref| <= max_rel * rms + 2^-8 |ref| elementwise and
    mean |o - ref| <= mean_rel * rms + mean(2^-9 |ref|).  A single bf16
    rounding (relative error up to 2^-9, 2^-8 across a rounding boundary) of
    an output near 10x the RMS already exceeds max_rel * rms on its own."""
    o, o_ref = _np(o), _np(o_ref)
    assert np.isfinite(o).all(), f"{what}: non-finite values"
    rms = np.sqrt(np.mean(o_ref ** 2))
    d = np.abs(o - o_ref)
    excess = d - (max_rel * rms + 2.0 ** -8 * np.abs(o_ref))
    assert excess.max() <= 0, f"{what}: worst excess {excess.max() / rms:.3e} rms"
    mean_bound = mean_rel * rms + np.mean(2.0 ** -9 * np.abs(o_ref))
    assert d.mean() <= mean_bound, f"{what}: mean {d.mean() / rms:.3e} rms"

