"""kda_chunk_fwd_host: the prefill on host buffers, the copies following the
rounds of the schedule.  It runs the same kernels on the same rounds as
kda_chunk_fwd, so its outputs and final state must equal the device entry
point's bit for bit: several overlapped rounds with a ragged tail and two
sequences, one round, no initial state, bf16 output, pinned and pageable
host memory, and the empty sequence."""
import pytest
import torch

from linear_attention_recurrence_fwd_gb300 import binding, build
from linear_attention_recurrence_fwd_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

KEYS = ("q", "k", "v", "log_alpha", "beta")


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    build.build()


@pytest.mark.parametrize("B,T,H,with_s0,out_dtype,pin", [
    (2, 9000, 3, True, torch.float32, True),     # overlapped rounds, ragged tail
    (1, 300, 2, True, torch.float32, True),      # one round
    (1, 8192, 2, False, torch.bfloat16, True),   # no initial state, bf16 output
    (1, 700, 2, True, torch.float32, False),     # pageable host memory
])
def test_host_entry_equals_device_entry(B, T, H, with_s0, out_dtype, pin):
    x = gen.make_inputs(B, T, H, 128, 128, seed=81, init_std=0.02)
    host = {k: (x[k].pin_memory() if pin else x[k].clone()) for k in KEYS}
    s0 = x["initial_state"] if with_s0 else None
    hs0 = (s0.pin_memory() if pin else s0.clone()) if s0 is not None else None
    out, fin = binding.kda_chunk_fwd_host(*[host[k] for k in KEYS], hs0, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert binding.kda_last_device_status() == 0
    g = {k: x[k].cuda() for k in KEYS}
    ref_out, ref_fin = binding.kda_chunk_fwd(*[g[k] for k in KEYS],
                                             None if s0 is None else s0.cuda(),
                                             out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out.cpu())
    assert torch.equal(fin, ref_fin.cpu())


def test_host_entry_empty_sequence_returns_the_initial_state():
    x = gen.make_inputs(1, 64, 2, 128, 128, seed=82, init_std=0.02)
    host = {k: x[k][:, :0].contiguous().pin_memory() for k in KEYS}
    s0 = x["initial_state"].pin_memory()
    out, fin = binding.kda_chunk_fwd_host(*[host[k] for k in KEYS], s0)
    torch.cuda.synchronize()
    assert out.shape == (1, 0, 2, 128)
    assert torch.equal(fin, x["initial_state"])
