"""Decode step on the GPU (through the C-ABI) against the fp64 oracle."""
import numpy as np
import pytest
import torch

from linear_attention_recurrence_fwd_gb300 import binding, build
from linear_attention_recurrence_fwd_gb300 import inputs as gen
from oracle import oracle as orc
from parity import (assert_bf16_output_close, assert_output_close, assert_state_close,
                    output_errors)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    build.build()


def _decode_inputs(N, H, seed, init_std=0.02, decay_mean=0.0):
    x = gen.make_inputs(N, 1, H, 128, 128, seed, decay_mean=decay_mean, init_std=init_std)
    sq = lambda t: t[:, 0].contiguous()
    return dict(q=sq(x["q"]), k=sq(x["k"]), v=sq(x["v"]), log_alpha=sq(x["log_alpha"]),
                beta=sq(x["beta"]), state=x["initial_state"])


def _gpu(x):
    return {k: v.cuda() for k, v in x.items()}


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_decode_one_step(out_dtype):
    x = _decode_inputs(8, 4, seed=11)
    d = _gpu(x)
    o = binding.kda_decode_step(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["state"],
                                out_dtype=out_dtype)
    torch.cuda.synchronize()
    ro, rs = orc.decode_step(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["state"])
    if out_dtype == torch.float32:
        assert_output_close(o, ro, 1e-5, 1e-6)
    else:
        assert_bf16_output_close(o, ro)
    assert_state_close(d["state"], rs, 1e-6)


def test_decode_chained_steps_and_scale():
    N, H, steps = 6, 2, 25
    xs = [_decode_inputs(N, H, seed=100 + s) for s in range(steps)]
    state = xs[0]["state"].clone()
    ref_state = state.double().numpy()
    dstate = state.cuda()
    for s in range(steps):
        d = _gpu({k: v for k, v in xs[s].items() if k != "state"})
        o = binding.kda_decode_step(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], dstate,
                                    scale=0.5, out_dtype=torch.float32)
        ro, ref_state = orc.decode_step(xs[s]["q"], xs[s]["k"], xs[s]["v"], xs[s]["log_alpha"],
                                        xs[s]["beta"], ref_state, scale=0.5)
        assert_output_close(o, ro, 1e-5, 1e-6, what=f"step {s}")
    assert_state_close(dstate, ref_state, 1e-5)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_decode_full_size_step(out_dtype):
    """256 sequences x 32 heads (the decode workload), one step, every output.
    bf16 outputs get the storage-rounding allowance: decode outputs have tails
    near 20x their RMS, where bf16's own rounding alone exceeds the max bar."""
    w = gen.WORKLOADS["decode"]
    x = _decode_inputs(w.B, w.H, seed=w.seed)
    d = _gpu(x)
    o = binding.kda_decode_step(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["state"],
                                out_dtype=out_dtype)
    torch.cuda.synchronize()
    ro, rs = orc.decode_step(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["state"])
    if out_dtype == torch.float32:
        assert_output_close(o, ro, 1e-5, 1e-6)
    else:
        assert_bf16_output_close(o, ro)
    assert_state_close(d["state"], rs)


def test_decode_zero_sequences_is_a_no_op():
    e = torch.empty((0, 2, 128), dtype=torch.bfloat16, device="cuda")
    st = torch.empty((0, 2, 128, 128), device="cuda")
    out = binding.kda_decode_step(e, e, e, e, torch.empty((0, 2), dtype=torch.bfloat16,
                                                          device="cuda"), st)
    assert out.shape == (0, 2, 128)
