"""Pins of the backward-pass oracle (kda_recurrence_bwd), CPU only.

The gradients are checked against things other than their own derivation:
central finite differences of the forward oracle (the C token loop), the
derivative autograd takes through an independent fp64 torch loop of the
forward recurrence, and a closed form (no write, no decay).  Each planted
mistake in the derivation must fail the finite-difference check.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as orc

NAMES = ("q", "k", "v", "log_alpha", "beta", "initial_state")


def _problem(seed, B=1, T=5, H=2, d=4, packed=None):
    rng = np.random.default_rng(seed)
    Ttot = sum(packed) if packed else T
    lead = (Ttot,) if packed else (B, T)
    n = len(packed) if packed else B
    q, k, v = (rng.standard_normal(lead + (H, d)) for _ in range(3))
    la = -5.0 / (1.0 + np.exp(-rng.standard_normal(lead + (H, d))))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(lead + (H,))))
    s0 = rng.standard_normal((n, H, d, d))
    d_out = rng.standard_normal(lead + (H, d))
    d_fin = rng.standard_normal((n, H, d, d))
    cu = None if packed is None else np.concatenate([[0], np.cumsum(packed)])
    return dict(q=q, k=k, v=v, log_alpha=la, beta=beta, initial_state=s0), d_out, d_fin, cu


def _loss(x, d_out, d_fin, cu, scale):
    o, f = orc.kda_recurrence(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                              x["initial_state"], scale=scale, cu_seqlens=cu)
    return float((o * d_out).sum() + (f * d_fin).sum())


def _finite_differences(x, d_out, d_fin, cu, scale, eps=1e-6):
    fd = {}
    for name in NAMES:
        arr = x[name]
        out = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            keep = arr[idx]
            arr[idx] = keep + eps
            lp = _loss(x, d_out, d_fin, cu, scale)
            arr[idx] = keep - eps
            lm = _loss(x, d_out, d_fin, cu, scale)
            arr[idx] = keep
            out[idx] = (lp - lm) / (2 * eps)
        fd[name] = out
    return fd


def _rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30))


@pytest.mark.parametrize("packed", [None, [3, 1, 4]], ids=["fixed", "packed"])
def test_gradients_match_finite_differences(packed):
    x, d_out, d_fin, cu = _problem(1, B=2, T=4, packed=packed)
    g = orc.kda_recurrence_bwd(*[x[n] for n in NAMES], d_out, d_fin, scale=0.7, cu_seqlens=cu)
    fd = _finite_differences(x, d_out, d_fin, cu, 0.7)
    for name in NAMES:
        assert _rel(g[name], fd[name]) < 1e-7, name


@pytest.mark.parametrize("mutation", [m for m in orc.BWD_MUTATIONS if m != "none"])
def test_planted_mistakes_are_caught(mutation):
    x, d_out, d_fin, cu = _problem(2, T=5)
    g = orc.kda_recurrence_bwd(*[x[n] for n in NAMES], d_out, d_fin, mutation=mutation)
    fd = _finite_differences(x, d_out, d_fin, cu, 1.0)
    assert max(_rel(g[name], fd[name]) for name in NAMES) > 1e-3


def _torch_loop(q, k, v, la, beta, s0, scale):
    """The forward recurrence as a plain fp64 torch loop, one sequence."""
    S = s0
    outs = []
    for t in range(q.shape[0]):
        Sp = torch.exp(la[t])[:, :, None] * S
        u = beta[t][:, None] * (v[t] - torch.einsum("hcv,hc->hv", Sp, k[t]))
        S = Sp + k[t][:, :, None] * u[:, None, :]
        outs.append(scale * torch.einsum("hcv,hc->hv", S, q[t]))
    return torch.stack(outs), S


def test_gradients_match_autograd():
    x, d_out, d_fin, _ = _problem(3, T=40, H=2, d=8)
    g = orc.kda_recurrence_bwd(*[x[n] for n in NAMES], d_out, d_fin, scale=0.5)
    tx = {n: torch.tensor(x[n][0] if n != "initial_state" else x[n][0], dtype=torch.float64,
                          requires_grad=True) for n in NAMES}
    o, f = _torch_loop(tx["q"], tx["k"], tx["v"], tx["log_alpha"], tx["beta"],
                       tx["initial_state"], 0.5)
    loss = (o * torch.tensor(d_out[0])).sum() + (f * torch.tensor(d_fin[0])).sum()
    loss.backward()
    for n in NAMES:
        ours = g[n][0]
        assert _rel(ours, tx[n].grad.numpy()) < 1e-11, n


def test_closed_form_without_write_or_decay():
    """beta = 0 and log_alpha = 0: the state stays S0, so o_t = scale S0^T q_t;
    dq_t = scale S0 do_t, dS0 = dF + scale sum_t q_t do_t^T, dk = dv = 0 and
    dlog_alpha_t = rowsum(G_t * S0) with G_t = dF + scale sum_{s >= t} q_s do_s^T."""
    x, d_out, d_fin, _ = _problem(4, T=6)
    x["beta"][:] = 0.0
    x["log_alpha"][:] = 0.0
    g = orc.kda_recurrence_bwd(*[x[n] for n in NAMES], d_out, d_fin, scale=0.3)
    S0, q, do, dF = x["initial_state"][0], x["q"][0], d_out[0], d_fin[0]
    outer = 0.3 * np.einsum("thc,thv->thcv", q, do)
    np.testing.assert_allclose(g["q"][0], 0.3 * np.einsum("hcv,thv->thc", S0, do), rtol=1e-13)
    np.testing.assert_allclose(g["initial_state"][0], dF + outer.sum(0), rtol=1e-12)
    assert np.abs(g["k"]).max() == 0 and np.abs(g["v"]).max() == 0
    tail = np.cumsum(outer[::-1], axis=0)[::-1]                    # sum over s >= t
    np.testing.assert_allclose(g["log_alpha"][0], np.einsum("thcv,hcv->thc", dF + tail, S0),
                               rtol=1e-12, atol=1e-12)
