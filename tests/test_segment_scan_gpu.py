"""The segment scan (kda_chunk_fwd_segments, and kda_chunk_fwd's own choice
for long sequences with few heads) against the fp64 oracle.

Each sequence is cut into segments of whole chunks; every segment's
cumulative transition and zero-start state are walked in parallel, composed
by a prefix scan into entry states, and the segments are walked once more
with outputs.  The results must meet the same bar as the unsegmented call,
for ragged segment splits, batches, d = 64, bf16 output, slow decay (the
state carries across every segment boundary), an in-place state, and a
length at which the walks run in overlapped rounds.
"""
import numpy as np
import pytest
import torch

from linear_attention_recurrence_fwd_gb300 import binding, build
from linear_attention_recurrence_fwd_gb300 import inputs as gen
from oracle import oracle as orc
from parity import assert_bf16_output_close, assert_output_close, assert_state_close

pytestmark = pytest.mark.gpu

KEYS = ("q", "k", "v", "log_alpha", "beta")


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    build.build()


def _check(B, T, H, d, segs, seed, slow=False, out_dtype=torch.float32, in_place=False):
    x = gen.make_inputs(B, T, H, d, d, seed, init_std=0.02)
    if slow:
        x["log_alpha"] = (x["log_alpha"].float() * 0.01).to(torch.bfloat16)
    g = {k: v.cuda() for k, v in x.items()}
    s0 = g["initial_state"].clone()
    fin = s0 if in_place else None
    out, fin = binding.kda_chunk_fwd_segments(*[g[k] for k in KEYS], s0, n_segments=segs,
                                              out_dtype=out_dtype, final_state=fin)
    torch.cuda.synchronize()
    assert binding.kda_last_device_status() == 0
    ro, rs = orc.kda_recurrence(*[x[k] for k in KEYS], x["initial_state"])
    if out_dtype == torch.float32:
        assert_output_close(out, ro, what=f"{segs} segments")
    else:
        assert_bf16_output_close(out, ro, what=f"{segs} segments")
    assert_state_close(fin, rs, what=f"{segs} segments")
    return out, fin, g


@pytest.mark.parametrize("segs", [2, 3, 5, 8])
def test_segments_against_oracle(segs):
    # 2000 tokens = 31 full chunks and a partial one: uneven segments
    _check(1, 2000, 2, 128, segs, seed=51)


def test_segments_batch_d64_bf16_output():
    _check(2, 777, 3, 64, 3, seed=52, out_dtype=torch.bfloat16)


def test_segments_slow_decay_in_place():
    _check(1, 1024, 2, 128, 4, seed=53, slow=True, in_place=True)


def test_segments_with_overlapped_rounds():
    # 3 segments of 128 chunks each: the walks run in rounds overlapped with
    # the intra-chunk stage of the next round
    _check(1, 3 * 128 * 64, 2, 128, 3, seed=54)


def test_one_segment_is_the_plain_call():
    x = gen.make_inputs(1, 500, 2, 128, 128, 55, init_std=0.02)
    g = {k: v.cuda() for k, v in x.items()}
    a, fa = binding.kda_chunk_fwd(*[g[k] for k in KEYS], g["initial_state"])
    b, fb = binding.kda_chunk_fwd_segments(*[g[k] for k in KEYS], g["initial_state"], n_segments=1)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(fa, fb)


def test_segments_close_to_unsegmented():
    """The scan reorders only the state pass's roundings: its results stay
    within a few 1e-4 of the RMS of the unsegmented call's."""
    out, fin, g = _check(1, 4096, 2, 128, 4, seed=56)
    a, fa = binding.kda_chunk_fwd(*[g[k] for k in KEYS], g["initial_state"])
    torch.cuda.synchronize()
    rms = a.double().pow(2).mean().sqrt().item()
    assert (out.double() - a.double()).abs().max().item() <= 2e-3 * rms
    assert_state_close(fin, fa.double().cpu().numpy(), 1e-3)


def test_long_sequences_with_few_heads_take_the_scan():
    """kda_chunk_fwd chooses the scan for the 1M-token, 16-head problem but not
    for the 64k, 32-head one.  Without the scan that call launches two
    kernels per round of its schedule; a scan adds its plan, combine and
    second-walk kernels, so its count is odd."""
    assert binding.kda_chunk_fwd_launches(1, 1 << 20, 16) % 2 == 1
    assert binding.kda_chunk_fwd_launches(1, 1 << 16, 32) % 2 == 0
