"""Failure detection, exercised without faulting the GPU.

* The decay-bound check (KDA_CHECK_DECAY, read once per process, so each case
  runs in a child process): a log-decay below -5 written on the host must set
  KDA_ERR_DECAY_BOUND in the device status word; valid inputs, or the check
  switched off, must not.
* A device wait that runs out on purpose (a barrier nothing arrives on, with
  a millisecond limit) must return KDA_ERR_TIMEOUT, free its TMEM and leave
  the context usable.
* Packed sequences whose offsets are inconsistent (longer than max_seqlen,
  past T_total, not starting at 0) must be flagged as invalid arguments and
  must not touch memory outside the caller's buffers.
* A workspace filled with NaN beforehand must not change any result (no
  kernel reads a workspace byte it did not write in the same call).
"""
import ctypes
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest
import torch

from linear_attention_recurrence_fwd_gb300 import binding, build
from linear_attention_recurrence_fwd_gb300 import inputs as gen
from oracle import oracle as orc
from parity import assert_output_close, assert_state_close

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = ("q", "k", "v", "log_alpha", "beta")


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    build.build()


def _child(body, check_decay):
    env = dict(os.environ)
    env.pop("KDA_CHECK_DECAY", None)
    if check_decay:
        env["KDA_CHECK_DECAY"] = "1"
    code = textwrap.dedent("""
        import sys, torch
        sys.path.insert(0, %r)
        from linear_attention_recurrence_fwd_gb300 import binding
        from linear_attention_recurrence_fwd_gb300 import inputs as gen
        x = gen.make_inputs(1, 300, 2, 128, 128, seed=5, init_std=0.02, device="cuda:0")
    """ % ROOT) + textwrap.dedent(body) + textwrap.dedent("""
        torch.cuda.synchronize()
        print("STATUS", binding.kda_last_device_status())
    """)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("STATUS")][-1]
    return int(line.split()[1])


CHUNK_CALL = """
    binding.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["initial_state"])
"""
VARLEN_CALL = """
    cu = torch.tensor([0, 100, 300], dtype=torch.int32, device="cuda:0")
    binding.kda_varlen_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], cu, 200, None)
"""
BAD_DECAY = """
    x["log_alpha"][0, 137, 1, 7] = -5.5
"""


@pytest.mark.parametrize("call", [CHUNK_CALL, VARLEN_CALL], ids=["chunk", "varlen"])
def test_decay_bound_flagged_when_checking(call):
    assert _child(BAD_DECAY + call, check_decay=True) == 5


@pytest.mark.parametrize("call", [CHUNK_CALL, VARLEN_CALL], ids=["chunk", "varlen"])
def test_decay_bound_quiet_on_valid_inputs(call):
    assert _child(call, check_decay=True) == 0


def test_decay_bound_not_checked_by_default():
    assert _child(BAD_DECAY + CHUNK_CALL, check_decay=False) == 0


def test_wait_that_runs_out_returns_timeout_and_frees_tmem():
    probe = binding.load_probe()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(3):  # TMEM freed each time, or the next allocation would stall
        st.zero_()
        assert probe.kda_probe_wait_timeout(1000, st.data_ptr(), stream) == 0
        torch.cuda.synchronize()
        assert st.item() == 6
    # the context is still usable: a prefill afterwards meets the bar
    x = gen.make_inputs(1, 200, 2, 128, 128, seed=21, init_std=0.02)
    g = {k: (v.cuda() if v is not None else None) for k, v in x.items()}
    out, fin = binding.kda_chunk_fwd(*[g[k] for k in KEYS], g["initial_state"])
    torch.cuda.synchronize()
    assert binding.kda_last_device_status() == 0
    ro, rs = orc.kda_recurrence(*[x[k] for k in KEYS], x["initial_state"])
    assert_output_close(out, ro)
    assert_state_close(fin, rs)


SENTINEL = 12345.0


def _varlen_slack(T_total, cu, max_seqlen, H=2, slack=128, seed=23):
    """Run kda_varlen_fwd on buffers followed by `slack` extra token rows
    (filled with a sentinel in the output) and return (out with slack, fin,
    status, inputs)."""
    x = gen.make_inputs(1, T_total + slack, H, 128, 128, seed=seed)
    g = {k: x[k][0].cuda() for k in KEYS}
    out = torch.full((T_total + slack, H, 128), SENTINEL, dtype=torch.float32, device="cuda")
    N = len(cu) - 1
    fin = torch.empty((N, H, 128, 128), dtype=torch.float32, device="cuda")
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    # the call sees only the first T_total rows of every token tensor
    binding.kda_varlen_fwd(*[g[k][:T_total] for k in KEYS], cu_d, max_seqlen, None,
                           out=out[:T_total], final_state=fin)
    torch.cuda.synchronize()
    return out, fin, binding.kda_last_device_status(), x


def test_varlen_sequence_longer_than_max_seqlen_is_flagged():
    out, fin, status, x = _varlen_slack(300, [0, 100, 300], max_seqlen=150)
    assert status == 1
    assert torch.isfinite(out[:250]).all()
    # the second sequence is clamped to 150 tokens: rows 250.. are never written
    assert (out[250:] == SENTINEL).all()
    # the first sequence (within the limit) is still right
    ro, rs = orc.kda_recurrence(*[x[k][0, :100] for k in KEYS], None,
                                cu_seqlens=np.array([0, 100]))
    assert_output_close(out[:100].cpu(), ro)
    assert_state_close(fin[0:1].cpu(), rs)


def test_varlen_offsets_past_the_end_touch_nothing_outside():
    # cu[N] = 460 > T_total = 300: clamped to the buffers, flagged
    out, fin, status, _ = _varlen_slack(300, [0, 120, 460], max_seqlen=400)
    assert status == 1
    assert (out[300:] == SENTINEL).all()
    assert torch.isfinite(out[:300]).all()


def test_varlen_offsets_not_starting_at_zero_are_flagged():
    out, fin, status, _ = _varlen_slack(300, [40, 120, 300], max_seqlen=300)
    assert status == 1
    assert (out[300:] == SENTINEL).all()


def test_varlen_decreasing_offsets_are_flagged():
    out, fin, status, _ = _varlen_slack(300, [0, 200, 100, 300], max_seqlen=300)
    assert status == 1
    assert (out[300:] == SENTINEL).all()


def _poisoned_call(lib, x, g, B, T, H):
    ws_bytes = lib.kda_chunk_fwd_workspace_size(B, T, H, 128, 128)
    ws = torch.full(((ws_bytes + 3) // 4,), float("nan"), dtype=torch.float32, device="cuda")
    out = torch.empty((B, T, H, 128), dtype=torch.float32, device="cuda")
    fin = torch.empty((B, H, 128, 128), dtype=torch.float32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = lib.kda_chunk_fwd(*[p(g[k]) for k in KEYS], p(g["initial_state"]), p(out), 1, p(fin),
                           B, T, H, 128, 128, 1.0, p(ws), ws.numel() * 4,
                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    assert binding.kda_last_device_status() == 0
    return out, fin


@pytest.mark.parametrize("B,T,H", [(2, 300, 3), (1, 8192, 2)], ids=["plain", "segmented"])
def test_nan_poisoned_workspace_changes_nothing(B, T, H):
    lib = binding.load()
    x = gen.make_inputs(B, T, H, 128, 128, seed=29, init_std=0.02)
    g = {k: v.cuda() for k, v in x.items()}
    out, fin = _poisoned_call(lib, x, g, B, T, H)
    ro, rs = orc.kda_recurrence(*[x[k] for k in KEYS], x["initial_state"])
    assert_output_close(out, ro)
    assert_state_close(fin, rs)
    ref_out, ref_fin = binding.kda_chunk_fwd(*[g[k] for k in KEYS], g["initial_state"])
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(fin, ref_fin)
