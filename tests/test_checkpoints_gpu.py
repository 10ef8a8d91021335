"""Prefill with state checkpoints (a prefix cache keeps the recurrent state at
fixed token boundaries): every checkpoint must equal the oracle's state after
that many tokens, and the outputs and final state must be exactly those of
the plain prefill."""
import pytest
import torch

from linear_attention_recurrence_fwd_gb300 import binding, build
from linear_attention_recurrence_fwd_gb300 import inputs as gen
from oracle import oracle as orc
from parity import assert_state_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    build.build()


def _oracle_states(x, every, n_ckpt):
    """State after every `every` tokens: the oracle run segment by segment,
    each from the previous segment's final state."""
    s = x["initial_state"]
    states = []
    for n in range(n_ckpt):
        seg = {k: x[k][:, n * every:(n + 1) * every] for k in ("q", "k", "v", "log_alpha", "beta")}
        _, s = orc.kda_recurrence(seg["q"], seg["k"], seg["v"], seg["log_alpha"], seg["beta"], s)
        states.append(s)
    return states


@pytest.mark.parametrize("B,T,H,every", [(2, 2148, 2, 512), (1, 700, 2, 64), (1, 8256, 2, 1024)])
def test_checkpoints_match_oracle(B, T, H, every):
    x = gen.make_inputs(B, T, H, 128, 128, seed=50 + every, init_std=0.02)
    g = {k: (v.cuda() if v is not None else None) for k, v in x.items()}
    args = [g[k] for k in ("q", "k", "v", "log_alpha", "beta")]
    out, fin, ck = binding.kda_chunk_fwd_checkpointed(*args, g["initial_state"],
                                                      checkpoint_every=every)
    ref_out, ref_fin = binding.kda_chunk_fwd(*args, g["initial_state"])
    torch.cuda.synchronize()
    assert binding.kda_last_device_status() == 0
    n_ckpt = T // every
    assert ck.shape == (B, n_ckpt, H, 128, 128)
    assert torch.equal(out, ref_out) and torch.equal(fin, ref_fin)
    for n, s in enumerate(_oracle_states(x, every, n_ckpt)):
        assert_state_close(ck[:, n], s, what=f"checkpoint {n}")


def test_no_checkpoint_when_shorter_than_interval():
    x = gen.make_inputs(1, 300, 2, 128, 128, seed=60, init_std=0.02)
    g = {k: (v.cuda() if v is not None else None) for k, v in x.items()}
    args = [g[k] for k in ("q", "k", "v", "log_alpha", "beta")]
    out, fin, ck = binding.kda_chunk_fwd_checkpointed(*args, g["initial_state"],
                                                      checkpoint_every=512)
    ref_out, ref_fin = binding.kda_chunk_fwd(*args, g["initial_state"])
    torch.cuda.synchronize()
    assert ck.shape[1] == 0
    assert torch.equal(out, ref_out) and torch.equal(fin, ref_fin)
