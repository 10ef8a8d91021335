"""Magnitudes away from the unit-variance synthetic inputs.

The state pass feeds 16-bit operands to the tensor cores (the state, the
corrected values and the chunk operators), so large values and small states
are checked against the oracle explicitly: values scaled by 300, an initial
state scaled by 1000, a small state (1e-4) with small values, and the same
under slow decay, where the state carries across many chunks and grows
largest.

The layer is linear in (v, initial state) jointly.  Scaling both by a power
of two must therefore scale every result by that power: the roundings are
the same ones wherever an intermediate stays a normal number, so only the
tiniest terms (16-bit subnormals) may differ, far below the bar.  That checks
the range directly, against the unscaled call.

With the initial state scaled by 1000 the first token's outputs reach ~60x
the RMS of all outputs.  A 16-bit operand carries a relative rounding of up
to 2^-11, so on those outputs the error is a few 1e-4 of their own size, a
few percent of the global RMS.  Such heavy-tailed cases are checked token by
token against the larger of the global RMS and the token's own RMS (the
mean error stays bound by the global RMS).
"""
import numpy as np
import pytest
import torch

from linear_attention_recurrence_fwd_gb300 import binding, build
from linear_attention_recurrence_fwd_gb300 import inputs as gen
from oracle import oracle as orc
from parity import MAX_REL, MEAN_REL, assert_output_close, assert_state_close

pytestmark = pytest.mark.gpu

KEYS = ("q", "k", "v", "log_alpha", "beta")


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    build.build()


def _scaled(v_scale, s_scale, seed, slow=False, T=1024, H=2):
    x = gen.make_inputs(1, T, H, 128, 128, seed, init_std=0.02)
    x["v"] = (x["v"].float() * v_scale).to(torch.bfloat16)
    x["initial_state"] = x["initial_state"] * s_scale
    if slow:  # log-decay -0.05 sigmoid(N(0,1)): the state lives across many chunks
        x["log_alpha"] = (x["log_alpha"].float() * 0.01).to(torch.bfloat16)
    return x


@pytest.mark.parametrize("v_scale,s_scale,slow", [
    (300.0, 1.0, False),
    (300.0, 1.0, True),
    (1.0, 1e3, False),
    (1.0, 1e3, True),
    (1e-4, 5e-3, False),   # a state of about 1e-4 and values of the same size
    (1e-4, 5e-3, True),
], ids=["v300", "v300-slow", "s1e3", "s1e3-slow", "small", "small-slow"])
def test_scaled_inputs_against_oracle(v_scale, s_scale, slow):
    x = _scaled(v_scale, s_scale, seed=41, slow=slow)
    g = {k: v.cuda() for k, v in x.items()}
    out, fin = binding.kda_chunk_fwd(*[g[k] for k in KEYS], g["initial_state"])
    torch.cuda.synchronize()
    assert binding.kda_last_device_status() == 0
    ro, rs = orc.kda_recurrence(*[x[k] for k in KEYS], x["initial_state"])
    if s_scale > 100:  # heavy-tailed outputs: each token against its own scale
        o = out.double().cpu().numpy()
        d = np.abs(o - ro)
        rms = np.sqrt(np.mean(ro ** 2))
        rms_t = np.sqrt(np.mean(ro ** 2, axis=(0, 2, 3)))
        worst = (d.max(axis=(0, 2, 3)) / np.maximum(rms, rms_t)).max()
        assert np.isfinite(o).all()
        assert worst <= MAX_REL, f"token-wise max {worst:.3e}"
        assert d.mean() / rms <= MEAN_REL, f"mean {d.mean() / rms:.3e}"
    else:
        assert_output_close(out, ro)
    assert_state_close(fin, rs)


@pytest.mark.parametrize("p2", [-6, 8, 12], ids=["x2^-6", "x2^8", "x2^12"])
def test_power_of_two_scaling_is_exact(p2):
    """(v, S0) -> (2^p v, 2^p S0) scales every output and the final state by
    2^p, to 1e-4 of the RMS (fp16 subnormals of the smallest v and state
    entries round differently at 2^-6).  |v| reaches ~2e4 at p = 12."""
    x = gen.make_inputs(1, 1000, 2, 128, 128, seed=43, init_std=0.02)
    g = {k: v.cuda() for k, v in x.items()}
    out, fin = binding.kda_chunk_fwd(*[g[k] for k in KEYS], g["initial_state"])
    f = 2.0 ** p2
    v2 = (g["v"].float() * f).to(torch.bfloat16)
    assert torch.equal(v2.float(), g["v"].float() * f)
    out2, fin2 = binding.kda_chunk_fwd(g["q"], g["k"], v2, g["log_alpha"], g["beta"],
                                       g["initial_state"] * f)
    torch.cuda.synchronize()
    assert binding.kda_last_device_status() == 0
    for a, b in ((out2, out), (fin2, fin)):
        assert torch.isfinite(a).all()
        rms = b.double().pow(2).mean().sqrt().item()
        err = (a.double() / f - b.double()).abs().max().item()
        assert err <= 1e-4 * rms, f"2^{p2}: max |scaled / 2^p - plain| = {err / rms:.3e} rms"


def test_values_beyond_the_fp16_range_are_flagged():
    """v scaled by 2^18 (|v| ~ 1e6): the delta-rule corrections leave the
    fp16 operand range, which the call reports as KDA_ERR_RANGE (8) instead
    of returning silently wrong results."""
    x = gen.make_inputs(1, 300, 2, 128, 128, seed=47, init_std=0.02)
    g = {k: v.cuda() for k, v in x.items()}
    v_big = (g["v"].float() * 2.0 ** 18).to(torch.bfloat16)
    binding.kda_chunk_fwd(g["q"], g["k"], v_big, g["log_alpha"], g["beta"], g["initial_state"])
    torch.cuda.synchronize()
    assert binding.kda_last_device_status() == 8
    # the flag is cleared by reading it; an in-range call reports nothing
    binding.kda_chunk_fwd(*[g[k] for k in KEYS], g["initial_state"])
    torch.cuda.synchronize()
    assert binding.kda_last_device_status() == 0
