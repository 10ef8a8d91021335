"""Records in a ring: a fixed-length call on the overlapped schedule whose
per-(chunk, head) records would pass 4 GiB keeps them for two segments only
(stage 1 of segment k + 2 starts after the state pass of segment k has
finished), so its workspace stops growing with T.

* The workspace of T = 65536 and of T = 122880 at 64 heads (both without
  the segment scan, both overlapped, 4.4 and 8.2 GB of records if kept
  whole) is the same, and under 1 GB.
* The T = 65536, 64-head call on the round schedule (the default for this
  many chains, and forced here with KDA_SCHEDULE=rounds), whose ring wraps
  four times, meets the oracle bar on every output and final-state element,
  and equals bit for bit the same call made through the default entry and
  through the one-segment entry point.
"""
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


def test_workspace_does_not_grow_with_T():
    lib = binding.load()
    a = lib.kda_chunk_fwd_workspace_size(1, 65536, 64, 128, 128)
    b = lib.kda_chunk_fwd_workspace_size(1, 122880, 64, 128, 128)
    assert a == b
    assert a < 1 << 30


def test_ring_that_wraps_against_oracle(monkeypatch):
    x = gen.make_inputs(1, 65536, 64, 128, 128, seed=71, init_std=0.02)
    g = {k: v.cuda() for k, v in x.items()}
    monkeypatch.setenv("KDA_SCHEDULE", "rounds")
    out, fin = binding.kda_chunk_fwd(*[g[k] for k in KEYS], g["initial_state"])
    torch.cuda.synchronize()
    assert binding.kda_last_device_status() == 0
    monkeypatch.delenv("KDA_SCHEDULE")
    # the default entry, and the one-segment entry point, make the same call
    out2, fin2 = binding.kda_chunk_fwd(*[g[k] for k in KEYS], g["initial_state"])
    torch.cuda.synchronize()
    assert binding.kda_last_device_status() == 0
    assert torch.equal(out, out2) and torch.equal(fin, fin2)
    del out2, fin2
    out2, fin2 = binding.kda_chunk_fwd_segments(*[g[k] for k in KEYS], g["initial_state"],
                                                n_segments=1)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(fin, fin2)
    o, f = out.cpu(), fin.cpu()
    del g, out, fin, out2, fin2
    torch.cuda.empty_cache()
    for h0 in range(0, 64, 16):  # 16 heads at a time bounds the oracle's host memory
        hs = slice(h0, h0 + 16)
        ro, rs = orc.kda_recurrence(*[x[k][:, :, hs] for k in KEYS], x["initial_state"][:, hs])
        assert_output_close(o[:, :, hs], ro, what=f"ringed call heads {h0}..")
        assert_state_close(f[:, hs], rs, what=f"ringed call state heads {h0}..")
