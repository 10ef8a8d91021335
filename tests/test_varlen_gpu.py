"""Packed (varlen) prefill on the GPU against the oracle and against
per-sequence fixed-length runs."""
import numpy as np
import pytest
import torch

from linear_attention_recurrence_fwd_gb300 import binding, build
from linear_attention_recurrence_fwd_gb300 import inputs as gen
from oracle import oracle as orc
from parity import assert_output_close, assert_state_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    build.build()


def _packed(lens, H, d, seed, init_std=0.02):
    x = gen.make_inputs(1, sum(lens), H, d, d, seed=seed, init_std=init_std,
                        n_states=len(lens))
    return x, gen.cu_seqlens_of(lens)


@pytest.mark.parametrize("lens", [[5, 64, 1, 90, 0, 130], [64, 64], [1], [200, 17, 300]])
def test_varlen_against_oracle(lens):
    x, cu = _packed(lens, 2, 128, seed=len(lens))
    g = {k: (v.cuda() if v is not None else None) for k, v in x.items()}
    out, fin = binding.kda_varlen_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"],
                                      cu.cuda(), max(lens), g["initial_state"],
                                      out_dtype=torch.float32)
    torch.cuda.synchronize()
    ro, rs = orc.kda_recurrence(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                x["initial_state"], cu_seqlens=cu.numpy())
    assert_output_close(out[0], ro)
    assert_state_close(fin, rs)


def test_varlen_equals_fixed_length_runs():
    lens = [70, 128, 33]
    x, cu = _packed(lens, 2, 128, seed=3)
    g = {k: (v.cuda() if v is not None else None) for k, v in x.items()}
    out, fin = binding.kda_varlen_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"],
                                      cu.cuda(), max(lens), g["initial_state"],
                                      out_dtype=torch.float32)
    for i, n in enumerate(lens):
        a, b = int(cu[i]), int(cu[i + 1])
        sl = lambda t: t[:, a:b].contiguous()
        oi, fi = binding.kda_chunk_fwd(sl(g["q"]), sl(g["k"]), sl(g["v"]), sl(g["log_alpha"]),
                                       sl(g["beta"]), g["initial_state"][i:i + 1].contiguous(),
                                       out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert torch.equal(oi[0], out[0, a:b]), f"sequence {i}"
        assert torch.equal(fi[0], fin[i])


def test_varlen_64k_workload_sampled_heads():
    """4 packed sequences summing to 65536 tokens, H=32; zero initial states.
    Every output of 4 of the 32 heads is compared (the oracle runs on those)."""
    w = gen.WORKLOADS["varlen_64k"]
    x = gen.workload_inputs(w)
    cu = gen.cu_seqlens_of(w.seqlens)
    g = {k: (v.cuda() if v is not None else None) for k, v in x.items()}
    out, fin = binding.kda_varlen_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"],
                                      cu.cuda(), max(w.seqlens), None)
    torch.cuda.synchronize()
    heads = [0, 9, 22, 31]
    sub = {k: x[k][:, :, heads] for k in ("q", "k", "v", "log_alpha", "beta")}
    ro, rs = orc.kda_recurrence(sub["q"], sub["k"], sub["v"], sub["log_alpha"], sub["beta"],
                                None, cu_seqlens=cu.numpy())
    o = out[0][:, heads]
    assert_output_close(o, ro)
    assert_state_close(fin[:, heads], rs)
