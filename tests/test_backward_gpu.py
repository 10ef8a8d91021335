"""kda_chunk_bwd (the backward of the prefill) against the fp64 oracle's
reverse-mode derivative, kda_recurrence_bwd.

Every gradient (q, k, v, log_alpha, beta and the initial state) is compared
element by element with the bar of tests/parity.py, each against its own
RMS: several chunks and a ragged tail, a single partial chunk, d = 64 with
two sequences, no initial state and no final-state gradient, slow decay (the
gradient carries across every chunk), scale != 1, tokens with beta = 0 (their
w comes from a column sum, the others' from the forward's u), the empty
sequence, 80 chains (no u from the forward), the 8k x 32-head problem the
bench times (three heads against the oracle) and the 64k x 32-head problem
(two heads).
"""
import numpy as np
import pytest
import torch

from linear_attention_recurrence_fwd_gb300 import binding, build
from linear_attention_recurrence_fwd_gb300 import inputs as gen
from oracle import oracle as orc
from parity import assert_output_close, assert_state_close

pytestmark = pytest.mark.gpu

KEYS = ("q", "k", "v", "log_alpha", "beta")
GRADS = ("q", "k", "v", "log_alpha", "beta")


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    build.build()


def _case(B, T, H, d, seed, with_s0=True, with_dfin=True, slow=False, scale=1.0,
          zero_beta=False):
    x = gen.make_inputs(B, T, H, d, d, seed, init_std=0.02)
    if slow:  # log-decay -0.05 sigmoid(N(0,1)): the gradient carries across every chunk
        x["log_alpha"] = (x["log_alpha"].float() * 0.01).to(torch.bfloat16)
    if zero_beta:  # every 7th token writes nothing (its dbeta still needs its w)
        x["beta"][:, ::7] = 0
    r = np.random.default_rng(seed + 1000)
    d_out = torch.from_numpy(r.standard_normal((B, T, H, d)).astype(np.float32))
    d_fin = torch.from_numpy((0.1 * r.standard_normal((B, H, d, d))).astype(np.float32))
    s0 = x["initial_state"] if with_s0 else None
    dfin = d_fin if with_dfin else None
    g = {k: x[k].cuda() for k in KEYS}
    got = binding.kda_chunk_bwd(*[g[k] for k in KEYS], d_out.cuda(),
                                initial_state=None if s0 is None else s0.cuda(),
                                d_final_state=None if dfin is None else dfin.cuda(), scale=scale)
    torch.cuda.synchronize()
    assert binding.kda_last_device_status() == 0
    ref = orc.kda_recurrence_bwd(*[x[k] for k in KEYS], s0, d_out, d_final=dfin, scale=scale)
    for name in GRADS:
        assert_output_close(got[name], ref[name], what=f"d{name}")
    assert_state_close(got["initial_state"], ref["initial_state"], what="d initial_state")
    return got, ref


def test_backward_several_chunks_ragged_tail():
    _case(1, 200, 2, 128, seed=61)


def test_backward_single_partial_chunk():
    _case(1, 37, 2, 128, seed=62)


def test_backward_head_dim_64_two_sequences():
    _case(2, 150, 3, 64, seed=63)


def test_backward_without_initial_state_or_final_gradient():
    _case(1, 130, 2, 128, seed=64, with_s0=False, with_dfin=False)


def test_backward_slow_decay_and_scale():
    _case(1, 320, 2, 128, seed=65, slow=True, scale=0.125)


def test_backward_tokens_with_zero_beta():
    _case(2, 200, 2, 128, seed=68, zero_beta=True)


def test_backward_many_chains_without_the_forward_u():
    """80 (sequence, head) chains: more than half the SMs, so the forward
    cannot leave u and every token's w takes the column sum."""
    _case(1, 130, 80, 128, seed=69)


def test_backward_empty_sequence_passes_the_final_gradient_through():
    x = gen.make_inputs(1, 64, 2, 128, 128, 66, init_std=0.02)
    g = {k: x[k][:, :0].contiguous().cuda() for k in KEYS}
    dfin = torch.randn(1, 2, 128, 128).cuda()
    got = binding.kda_chunk_bwd(*[g[k] for k in KEYS], torch.empty(1, 0, 2, 128).cuda(),
                                initial_state=x["initial_state"].cuda(), d_final_state=dfin)
    torch.cuda.synchronize()
    assert torch.equal(got["initial_state"], dfin)


def test_backward_equals_autograd_of_the_forward_on_a_tiny_case():
    """The same gradients as torch autograd through the oracle-independent
    token loop written here in plain torch fp64 (a second derivation: the
    backward kernel must agree with differentiating the forward itself)."""
    B, T, H, d = 1, 70, 1, 128
    x = gen.make_inputs(B, T, H, d, d, 67, init_std=0.02)
    leaf = {k: x[k].double().requires_grad_(True) for k in KEYS}
    s0 = x["initial_state"].double().requires_grad_(True)
    S = s0[0, 0]
    outs = []
    for t in range(T):
        a = torch.exp(leaf["log_alpha"][0, t, 0])
        Sp = a[:, None] * S
        u = leaf["beta"][0, t, 0] * (leaf["v"][0, t, 0] - Sp.T @ leaf["k"][0, t, 0])
        S = Sp + torch.outer(leaf["k"][0, t, 0], u)
        outs.append(S.T @ leaf["q"][0, t, 0])
    out = torch.stack(outs)
    d_out = torch.randn(T, d, dtype=torch.float64, generator=torch.Generator().manual_seed(7))
    ((out * d_out).sum()).backward()
    g = {k: x[k].cuda() for k in KEYS}
    got = binding.kda_chunk_bwd(*[g[k] for k in KEYS], d_out.float().reshape(B, T, H, d).cuda(),
                                initial_state=x["initial_state"].cuda())
    torch.cuda.synchronize()
    for name in GRADS:
        assert_output_close(got[name], leaf[name].grad, what=f"d{name} vs autograd")
    assert_state_close(got["initial_state"], s0.grad, what="d initial_state vs autograd")


def test_backward_of_the_8k_bench_problem_on_sampled_heads():
    """The configuration the bench times (B=1, T=8192, H=32, the prefill_8k
    inputs and seed, random d_out): every head is computed on the GPU; three
    heads (first, a middle one, last) are compared with the oracle in full
    (heads are independent, so the oracle takes only those)."""
    w = gen.WORKLOADS["prefill_8k"]
    x = gen.workload_inputs(w)
    r = np.random.default_rng(w.seed + 2)
    d_out = torch.from_numpy(r.standard_normal((w.B, w.T, w.H, w.dv)).astype(np.float32))
    g = {k: x[k].cuda() for k in KEYS}
    got = binding.kda_chunk_bwd(*[g[k] for k in KEYS], d_out.cuda(),
                                initial_state=x["initial_state"].cuda())
    torch.cuda.synchronize()
    assert binding.kda_last_device_status() == 0
    got = {k: (v.cpu() if v is not None else None) for k, v in got.items()}
    for h in (0, 17, 31):
        hs = slice(h, h + 1)
        ref = orc.kda_recurrence_bwd(*[x[k][:, :, hs] for k in KEYS], x["initial_state"][:, hs],
                                     d_out[:, :, hs])
        for name in GRADS:
            assert_output_close(got[name][:, :, hs], ref[name], what=f"d{name} head {h}")
        assert_state_close(got["initial_state"][:, hs], ref["initial_state"],
                           what=f"d initial_state head {h}")


def test_backward_of_the_64k_problem_on_sampled_heads():
    """Training at 64k contexts (the studioglobal.ai page, section "Grosse
    Kapazitaet..."): the T = 65536, H = 32 problem of the prefill bench
    (its inputs and seed, random d_out), every head computed on the GPU, two
    heads (first and last) compared with the oracle in full."""
    w = gen.WORKLOADS["prefill_64k"]
    x = gen.workload_inputs(w)
    r = np.random.default_rng(w.seed + 2)
    d_out = torch.from_numpy(r.standard_normal((w.B, w.T, w.H, w.dv)).astype(np.float32))
    g = {k: x[k].cuda() for k in KEYS}
    got = binding.kda_chunk_bwd(*[g[k] for k in KEYS], d_out.cuda(),
                                initial_state=x["initial_state"].cuda())
    torch.cuda.synchronize()
    assert binding.kda_last_device_status() == 0
    for h in (0, 31):
        hs = slice(h, h + 1)
        ref = orc.kda_recurrence_bwd(*[x[k][:, :, hs] for k in KEYS], x["initial_state"][:, hs],
                                     d_out[:, :, hs])
        for name in GRADS:
            assert_output_close(got[name][:, :, hs].cpu(), ref[name], what=f"d{name} head {h}")
        assert_state_close(got["initial_state"][:, hs].cpu(), ref["initial_state"],
                           what=f"d initial_state head {h}")
