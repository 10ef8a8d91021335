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


def test_noalloc_matches_workspace_entry_point(cuda_device):
    build.build()
    lib = binding.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for seed, (B, T, H) in ((31, (1, 300, 3)), (32, (2, 190, 4))):
        x = gen.make_inputs(B, T, H, 128, 128, seed, init_std=0.02, device=cuda_device)
        args = [x[k] for k in ("q", "k", "v", "log_alpha", "beta")]
        ref_out, ref_fin = binding.kda_chunk_fwd(*args, x["initial_state"])
        out = torch.full_like(ref_out, float("nan"))
        fin = torch.full_like(ref_fin, float("nan"))
        rc = lib.kda_chunk_fwd_noalloc(*[_ptr(a) for a in args], _ptr(x["initial_state"]),
                                       _ptr(out), 1, _ptr(fin), B, T, H, 128, 128, 1.0, stream)
        assert rc == 0, binding.kda_status_string(rc)
        torch.cuda.synchronize()
        assert_output_close(out, ref_out.double().cpu().numpy(), 1e-6, 1e-7, what=f"seed {seed}")
        assert_state_close(fin, ref_fin.double().cpu().numpy(), 1e-6, what=f"seed {seed}")


def test_noalloc_rejects_problems_beyond_its_scratch(cuda_device):
    lib = binding.load()
    f = ctypes.c_void_p(16)
    # 1 * ceil(4096 / 64) * 32 = 2048 records > 1008: refused before any launch
    rc = lib.kda_chunk_fwd_noalloc(f, f, f, f, f, None, f, 1, None, 1, 4096, 32, 128, 128, 1.0,
                                   None)
    assert rc == 7
