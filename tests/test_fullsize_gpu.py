"""The named workloads against the fp64 oracle at full size, every head.

* prefill_64k: B=1, T=65536, H=32, d=128, random fp32 initial state (the
  benchmark's headline problem, same seed, same launch configuration; the
  fused launch forced on it gives the same bits);
* varlen_64k: four packed sequences summing to 65536 tokens, H=32;
* long_1m: B=1, T=1,048,576, H=16, decay concentrated near the bound, through
  the segment scan kda_chunk_fwd picks and again in one fused launch without it;
* decode: 256 sequences x 32 heads from the 64-set input pool, 128 chained
  in-place steps (step s uses set s mod 64), every step's output compared.

Every output element and every final-state element is compared with the
bar of tests/parity.py (fp32 outputs).  The oracle runs on the host cores;
the long-context problem is checked two heads at a time to bound host
memory (the oracle converts its inputs to fp64).
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


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    build.build()


def _status_ok():
    st = binding.kda_last_device_status()
    assert st == 0, binding.kda_status_string(st)


def test_prefill_64k_all_heads_against_oracle(monkeypatch):
    w = gen.WORKLOADS["prefill_64k"]
    dev = torch.device("cuda:0")
    x = gen.workload_inputs(w, device=dev)
    out, fin = binding.kda_chunk_fwd(*[x[k] for k in KEYS], x["initial_state"],
                                     out_dtype=torch.float32)
    torch.cuda.synchronize()
    _status_ok()
    # the same call on the fused launch (which this shape does not take by
    # itself): the same arithmetic, bit for bit
    monkeypatch.setenv("KDA_SCHEDULE", "fused")
    out2, fin2 = binding.kda_chunk_fwd(*[x[k] for k in KEYS], x["initial_state"],
                                       out_dtype=torch.float32)
    torch.cuda.synchronize()
    monkeypatch.delenv("KDA_SCHEDULE")
    _status_ok()
    assert torch.equal(out, out2) and torch.equal(fin, fin2)
    del out2, fin2
    host = {k: x[k].cpu() for k in KEYS}
    s0 = x["initial_state"].cpu()
    o, s = out.cpu(), fin.cpu()
    del x, out, fin
    torch.cuda.empty_cache()
    ro, rs = orc.kda_recurrence(*[host[k] for k in KEYS], s0)
    assert_output_close(o, ro, what="prefill_64k out")
    assert_state_close(s, rs, what="prefill_64k state")
    # every head on its own meets the bar too (a head-local fault cannot hide
    # behind the other heads' RMS)
    for h in range(w.H):
        assert_output_close(o[:, :, h], ro[:, :, h], what=f"prefill_64k head {h}")
        assert_state_close(s[:, h], rs[:, h], what=f"prefill_64k head {h} state")


def test_varlen_64k_all_heads_against_oracle():
    w = gen.WORKLOADS["varlen_64k"]
    dev = torch.device("cuda:0")
    x = gen.workload_inputs(w, device=dev)
    cu = gen.cu_seqlens_of(w.seqlens)
    out, fin = binding.kda_varlen_fwd(*[x[k] for k in KEYS], cu.to(dev), max(w.seqlens), None,
                                      out_dtype=torch.float32)
    torch.cuda.synchronize()
    _status_ok()
    host = {k: x[k].cpu() for k in KEYS}
    o, s = out.cpu(), fin.cpu()
    del x, out, fin
    torch.cuda.empty_cache()
    ro, rs = orc.kda_recurrence(*[host[k] for k in KEYS], None, cu_seqlens=cu.numpy())
    assert_output_close(o[0], ro, what="varlen_64k out")
    assert_state_close(s, rs, what="varlen_64k state")
    for n in range(len(w.seqlens)):
        a, b = int(cu[n]), int(cu[n + 1])
        assert_output_close(o[0, a:b], ro[a:b], what=f"varlen_64k sequence {n}")
        assert_state_close(s[n], rs[n], what=f"varlen_64k sequence {n} state")


def test_long_1m_all_heads_against_oracle():
    w = gen.WORKLOADS["long_1m"]
    dev = torch.device("cuda:0")
    x = gen.workload_inputs(w, device=dev)
    out, fin = binding.kda_chunk_fwd(*[x[k] for k in KEYS], None, out_dtype=torch.float32)
    torch.cuda.synchronize()
    _status_ok()
    o, s = out.cpu(), fin.cpu()
    del out, fin
    # without the scan: one fused launch, 16 chains whose rings of 16
    # records wrap a thousand times
    out, fin = binding.kda_chunk_fwd_segments(*[x[k] for k in KEYS], None, n_segments=1,
                                              out_dtype=torch.float32)
    torch.cuda.synchronize()
    _status_ok()
    o1, s1 = out.cpu(), fin.cpu()
    host = {k: x[k].cpu() for k in KEYS}
    del x, out, fin
    torch.cuda.empty_cache()
    for h0 in range(0, w.H, 2):
        hs = slice(h0, h0 + 2)
        ro, rs = orc.kda_recurrence(*[host[k][:, :, hs] for k in KEYS], None)
        assert_output_close(o[:, :, hs], ro, what=f"long_1m heads {h0}-{h0 + 1}")
        assert_state_close(s[:, hs], rs, what=f"long_1m heads {h0}-{h0 + 1} state")
        assert_output_close(o1[:, :, hs], ro, what=f"long_1m fused heads {h0}-{h0 + 1}")
        assert_state_close(s1[:, hs], rs, what=f"long_1m fused heads {h0}-{h0 + 1} state")
        del ro, rs


def test_decode_256x32_chained_steps_against_oracle():
    """128 in-place steps of the decode workload; step s uses input set s mod 64
    of the pool.  The chain of steps is one 128-token sequence per (sequence,
    head) for the oracle, so every step's output and the final state are
    compared with the token-by-token recurrence."""
    w = gen.WORKLOADS["decode"]
    dev = torch.device("cuda:0")
    pool, steps = 64, 128
    xd = gen.make_inputs(w.B, pool, w.H, 128, 128, w.seed, init_std=w.init_std, device=dev)
    sets = [[xd[k][:, s].contiguous() for k in KEYS] for s in range(pool)]
    state = xd["initial_state"].clone()
    s0 = xd["initial_state"].cpu()
    outs = torch.empty((w.B, steps, w.H, 128), dtype=torch.float32, device=dev)
    for s in range(steps):
        outs[:, s].copy_(binding.kda_decode_step(*sets[s % pool], state))
    torch.cuda.synchronize()
    idx = torch.arange(steps, device=dev) % pool
    seq = {k: xd[k][:, idx].cpu() for k in KEYS}
    ro, rs = orc.kda_recurrence(*[seq[k] for k in KEYS], s0)
    o = outs.cpu()
    for s in range(steps):
        assert_output_close(o[:, s], ro[:, s], what=f"decode step {s}")
    assert_state_close(state, rs, what="decode state after 128 steps")
