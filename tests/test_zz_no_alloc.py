"""The allocation-free prefill entry point (kda_chunk_fwd_noalloc) against the
workspace-taking one, through the C ABI.

It exists for callers that may not allocate device memory themselves, so it
keeps its intermediates in a fixed device array inside the library.  Two
calls in a row with different inputs check that the shared scratch, which
keeps the previous call's contents, does not leak into the next result.
This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""
import ctypes

import pytest
import torch

from linear_attention_recurrence_fwd_gb300 import binding, build
from linear_attention_recurrence_fwd_gb300 import inputs as gen
from parity import assert_output_close, assert_state_close

pytestmark = pytest.mark.gpu


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


# The most (chunk, head) records the fixed scratch holds (include/kda.h).
MAX_RECORDS = 1008


def _two_calls(lib, cases, d=128, out_dtype=torch.float32):
    """Each case through kda_chunk_fwd_noalloc, back to back (the second call
    finds the first call's records in the shared scratch), against
    kda_chunk_fwd on the same inputs."""
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    code = 1 if out_dtype == torch.float32 else 0
    for seed, (B, T, H) in cases:
        x = gen.make_inputs(B, T, H, d, d, seed, init_std=0.02, device="cuda:0")
        args = [x[k] for k in ("q", "k", "v", "log_alpha", "beta")]
        ref_out, ref_fin = binding.kda_chunk_fwd(*args, x["initial_state"], out_dtype=out_dtype)
        out = torch.full_like(ref_out, float("nan"))
        fin = torch.full_like(ref_fin, float("nan"))
        rc = lib.kda_chunk_fwd_noalloc(*[_ptr(a) for a in args], _ptr(x["initial_state"]),
                                       _ptr(out), code, _ptr(fin), B, T, H, d, d, 1.0, stream)
        assert rc == 0, binding.kda_status_string(rc)
        torch.cuda.synchronize()
        assert binding.kda_last_device_status() == 0
        assert_output_close(out.float(), ref_out.float().double().cpu().numpy(), 1e-6, 1e-7,
                            what=f"seed {seed}")
        assert_state_close(fin, ref_fin.double().cpu().numpy(), 1e-6, what=f"seed {seed}")


def test_noalloc_matches_workspace_entry_point(cuda_device):
    build.build()
    _two_calls(binding.load(), ((31, (1, 300, 3)), (32, (2, 190, 4))))


def test_noalloc_at_its_record_limit(cuda_device):
    """Exactly the documented maximum: the last record ends near the end of
    the scratch array.  A smaller call follows, so stale records from the
    large one would show."""
    build.build()
    T = 64 * (MAX_RECORDS // 16)
    assert (T // 64) * 16 == MAX_RECORDS
    _two_calls(binding.load(), ((33, (1, T, 16)), (34, (1, 333, 2))))


def test_noalloc_head_dim_64_bf16_output(cuda_device):
    build.build()
    _two_calls(binding.load(), ((35, (2, 250, 3)), (36, (1, 129, 5))), d=64,
               out_dtype=torch.bfloat16)

