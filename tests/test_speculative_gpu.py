"""Speculative-decoding pair: verify computes the outputs of K drafted tokens
from a state it only reads; commit advances the state by each sequence's
accepted count from the same cached inputs.  Checked against the fp64
oracle (the recurrence over the drafted tokens) and against chained
single-token decode steps."""
import numpy as np
import pytest
import torch

from linear_attention_recurrence_fwd_gb300 import binding, build
from linear_attention_recurrence_fwd_gb300 import inputs as gen
from oracle import oracle as orc
from parity import assert_bf16_output_close, assert_output_close, assert_state_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    build.build()


def _draft(N, K, H, seed):
    # N sequences of K draft tokens: [N, K, H, d] is the [B, T, H, d] layout with T = K
    return gen.make_inputs(N, K, H, 128, 128, seed=seed, init_std=0.02)


# K = 19 stages the drafted tokens in several passes, the last one ragged
@pytest.mark.parametrize("N,K,H,out_dtype", [(5, 4, 3, torch.float32), (8, 7, 2, torch.bfloat16),
                                              (3, 1, 2, torch.float32), (3, 19, 2, torch.float32)])
def test_verify_matches_oracle_and_leaves_state(N, K, H, out_dtype):
    x = _draft(N, K, H, seed=70 + K)
    g = {k: v.cuda() for k, v in x.items()}
    s = g["initial_state"].clone()
    out = binding.kda_decode_verify(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"], s,
                                    scale=0.8, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert torch.equal(s, g["initial_state"])  # only read
    ro, _ = orc.kda_recurrence(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                               x["initial_state"], scale=0.8)
    if out_dtype == torch.bfloat16:
        assert_bf16_output_close(out, ro)
    else:
        assert_output_close(out, ro)


# counts above K are clamped to K; with K = 13 the accepted counts end inside
# staging passes and on their boundaries
@pytest.mark.parametrize("K,acc", [(5, [0, 1, 2, 5, 3, 9]), (13, [0, 8, 9, 13, 20, 4])])
def test_commit_matches_oracle_per_accepted_count(K, acc):
    N, H = 6, 2
    x = _draft(N, K, H, seed=80 + K)
    g = {k: v.cuda() for k, v in x.items()}
    acc = np.array(acc, dtype=np.int32)
    s = g["initial_state"].clone()
    binding.kda_decode_commit(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"], s,
                              torch.from_numpy(acc).cuda())
    torch.cuda.synchronize()
    for n in range(N):
        m = min(int(acc[n]), K)
        if m == 0:
            assert torch.equal(s[n], g["initial_state"][n])
            continue
        sub = {k: x[k][n:n + 1, :m] for k in ("q", "k", "v", "log_alpha", "beta")}
        _, rs = orc.kda_recurrence(sub["q"], sub["k"], sub["v"], sub["log_alpha"], sub["beta"],
                                   x["initial_state"][n:n + 1])
        assert_state_close(s[n:n + 1], rs, what=f"sequence {n}, {m} accepted")


def test_verify_then_commit_equals_decode_steps():
    """verify's outputs and commit's state are those of chained decode steps."""
    N, K, H = 4, 3, 2
    x = _draft(N, K, H, seed=90)
    g = {k: v.cuda() for k, v in x.items()}
    out = binding.kda_decode_verify(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"],
                                    g["initial_state"])
    s_step = g["initial_state"].clone()
    for t in range(K):
        o_t = binding.kda_decode_step(*(g[k][:, t].contiguous() for k in
                                        ("q", "k", "v", "log_alpha", "beta")), s_step)
        torch.cuda.synchronize()
        assert torch.allclose(out[:, t], o_t, rtol=1e-5, atol=1e-6)
    s = g["initial_state"].clone()
    binding.kda_decode_commit(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"], s,
                              torch.full((N,), K, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert torch.allclose(s, s_step, rtol=1e-5, atol=1e-6)
