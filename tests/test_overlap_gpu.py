"""The two schedules of a long prefill with few (sequence, head) states.

* Fused (fixed lengths, the default): one cooperative launch in which some
  CTAs walk the state chains while the others run the intra-chunk stage in
  chunk order into a ring of records.
* Rounds (packed sequences, the ablation, host-buffer calls, or
  KDA_SCHEDULE=rounds): segments whose intra-chunk stage overlaps the
  previous segment's state pass, with the state carried between segments.

Every variant is checked against the fp64 oracle under both schedules where
both apply: several sequences, packed sequences of unequal length (some
shorter than a segment, one empty), bf16 output, d = 64, an in-place state
and the per-pair diagonal ablation; and the two schedules agree bit for bit.
"""
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


def _cuda(x):
    return {k: (v.cuda() if v is not None else None) for k, v in x.items()}


def _ref(x, **kw):
    return orc.kda_recurrence(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                              x["initial_state"], **kw)


@pytest.fixture(params=["fused", "rounds"])
def schedule(request, monkeypatch):
    if request.param == "rounds":
        monkeypatch.setenv("KDA_SCHEDULE", "rounds")
    else:
        monkeypatch.delenv("KDA_SCHEDULE", raising=False)
    return request.param


def test_schedules(monkeypatch):
    # the cases below only test what they claim if these fixed-length shapes
    # take one fused launch (few chains; 32 of them up to 512 chunks), the
    # 32-head 64k problem the segmented schedule, and with
    # KDA_SCHEDULE=rounds every shape the segmented schedule (2 launches per
    # segment) from 128 chunks on
    monkeypatch.delenv("KDA_SCHEDULE", raising=False)
    for shape in ((2, 9000, 2), (1, 8192, 32), (1, 4096, 2), (1, 65536, 16)):
        assert binding.kda_chunk_fwd_launches(*shape) == 1
    assert binding.kda_chunk_fwd_launches(1, 65536, 32) > 2
    monkeypatch.setenv("KDA_SCHEDULE", "rounds")
    assert binding.kda_chunk_fwd_launches(2, 9000, 2) > 2
    assert binding.kda_chunk_fwd_launches(1, 8192, 32) > 2
    assert binding.kda_chunk_fwd_launches(1, 4096, 2) == 2


@pytest.mark.parametrize("d,out_dtype,B,T,H,forced", [(128, torch.float32, 2, 9000, 2, "auto"),
                                                      (64, torch.bfloat16, 2, 9000, 2, "auto"),
                                                      (128, torch.float32, 1, 8192, 64, "fused")])
def test_fused_equals_rounds(monkeypatch, d, out_dtype, B, T, H, forced):
    """The same arithmetic per item and per chunk under either schedule (64
    chains: a fused launch that KDA_SCHEDULE=fused forces, half the SMs on
    chains)."""
    if forced == "fused":
        monkeypatch.setenv("KDA_SCHEDULE", "fused")
        assert binding.kda_chunk_fwd_launches(B, T, H) == 1
    x = gen.make_inputs(B, T, H, d, d, seed=46, init_std=0.02)
    g = _cuda(x)
    res = []
    for sched in ("fused", "rounds"):
        if sched == "rounds":
            monkeypatch.setenv("KDA_SCHEDULE", "rounds")
        elif forced == "fused":
            monkeypatch.setenv("KDA_SCHEDULE", "fused")
        else:
            monkeypatch.delenv("KDA_SCHEDULE", raising=False)
        out, fin = binding.kda_chunk_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"],
                                         g["initial_state"], scale=0.9, out_dtype=out_dtype)
        torch.cuda.synchronize()
        assert binding.kda_last_device_status() == 0
        res.append((out, fin))
    assert torch.equal(res[0][0], res[1][0]) and torch.equal(res[0][1], res[1][1])


@pytest.mark.parametrize("d,out_dtype", [(128, torch.float32), (64, torch.bfloat16)])
def test_overlap_batch_of_sequences(schedule, d, out_dtype):
    x = gen.make_inputs(2, 9000, 2, d, d, seed=41, init_std=0.02)
    g = _cuda(x)
    out, fin = binding.kda_chunk_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"],
                                     g["initial_state"], scale=0.9, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert binding.kda_last_device_status() == 0
    ro, rs = _ref(x, scale=0.9)
    if out_dtype == torch.bfloat16:
        assert_bf16_output_close(out, ro)
    else:
        assert_output_close(out, ro)
    assert_state_close(fin, rs)


def test_overlap_in_place_state(schedule):
    x = gen.make_inputs(1, 8300, 2, 128, 128, seed=42, init_std=0.02)
    g = _cuda(x)
    s = g["initial_state"].clone()
    out, _ = binding.kda_chunk_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"], s,
                                   final_state=s)
    torch.cuda.synchronize()
    ro, rs = _ref(x)
    assert_output_close(out, ro)
    assert_state_close(s, rs)


def test_overlap_packed_sequences():
    lens = [9000, 300, 0, 12345, 64]
    x = gen.make_inputs(1, sum(lens), 2, 128, 128, seed=43, init_std=0.02, n_states=len(lens))
    cu = gen.cu_seqlens_of(lens)
    g = _cuda(x)
    out, fin = binding.kda_varlen_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"],
                                      cu.cuda(), max(lens), g["initial_state"])
    torch.cuda.synchronize()
    assert binding.kda_last_device_status() == 0
    ro, rs = orc.kda_recurrence(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                x["initial_state"], cu_seqlens=cu.numpy())
    assert_output_close(out[0], ro)
    assert_state_close(fin, rs)


def test_overlap_diag_per_pair_ablation(monkeypatch):
    x = gen.make_inputs(1, 8192, 2, 128, 128, seed=44, init_std=0.02)
    g = _cuda(x)
    monkeypatch.setenv("KDA_ABLATE_DIAG", "1")
    out, fin = binding.kda_chunk_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"],
                                     g["initial_state"])
    torch.cuda.synchronize()
    monkeypatch.delenv("KDA_ABLATE_DIAG")
    ro, rs = _ref(x)
    assert_output_close(out, ro)
    assert_state_close(fin, rs)


def test_overlap_repeated_calls_are_identical(schedule):
    """The item counters and ring flags start over: back-to-back calls agree bit for bit."""
    x = gen.make_inputs(1, 8192, 2, 128, 128, seed=45, init_std=0.02)
    g = _cuda(x)
    outs = []
    for _ in range(3):
        o, f = binding.kda_chunk_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"],
                                     g["initial_state"])
        outs.append((o.clone(), f.clone()))
    torch.cuda.synchronize()
    for o, f in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(f, outs[0][1])
