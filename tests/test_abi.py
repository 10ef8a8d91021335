"""The C-ABI library loads, exports every symbol its headers declare, and
rejects bad arguments synchronously (no GPU needed: validation runs before
any CUDA call)."""
import ctypes
import os
import re

import pytest

from linear_attention_recurrence_fwd_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def _declared(header):
    text = open(os.path.join(ROOT, "include", header)).read()
    return re.findall(r"^KDA_API\s+[\w\s\*]+?\b(kda_\w+)\s*\(", text, flags=re.M)


@pytest.mark.parametrize("header,path", [("kda.h", binding.LIB_PATH),
                                         ("kda_probe.h", binding.PROBE_LIB_PATH)])
def test_every_declared_symbol_is_exported(lib, header, path):
    names = _declared(header)
    assert names, header
    so = ctypes.CDLL(path)
    for n in names:
        assert hasattr(so, n), f"{n} declared in {header} but not exported by {path}"


def test_binding_covers_the_product_header(lib):
    assert sorted(_declared("kda.h")) == sorted(binding.EXPORTS)


def test_status_strings(lib):
    for code, text in binding.STATUS.items():
        assert binding.kda_status_string(code) == text
    assert "sm_103a" in binding.kda_version()


F = ctypes.c_void_p(16)      # aligned fake pointer: never dereferenced on these paths
MIS = ctypes.c_void_p(18)    # misaligned


def _chunk(lib, q=F, out=F, B=1, T=64, H=2, dk=128, dv=128, dt=0, s0=None):
    return lib.kda_chunk_fwd(q, F, F, F, F, s0, out, dt, None, B, T, H, dk, dv, 1.0, None, 0, None)


def test_chunk_argument_errors(lib):
    assert _chunk(lib, q=None) == 1
    assert _chunk(lib, out=None) == 1
    assert _chunk(lib, B=-1) == 1
    assert _chunk(lib, H=0) == 1
    assert _chunk(lib, dk=96, dv=96) == 2
    assert _chunk(lib, dk=128, dv=64) == 2
    assert _chunk(lib, dt=7) == 2
    assert _chunk(lib, q=MIS) == 3
    assert _chunk(lib, s0=MIS) == 3


def test_varlen_argument_errors(lib):
    call = lambda cu=F, N=2, Tt=10, mx=8, dk=128: lib.kda_varlen_fwd(
        F, F, F, F, F, cu, N, Tt, mx, None, F, 0, None, 2, dk, dk, 1.0, None, 0, None)
    assert call(cu=None) == 1
    assert call(N=-1) == 1
    assert call(mx=0) == 1
    assert call(cu=MIS) == 3
    assert call(dk=32) == 2


def test_decode_argument_errors(lib):
    call = lambda st=F, N=4, dk=128, dt=0: lib.kda_decode_step(
        F, F, F, F, F, st, F, dt, N, 2, dk, dk, 1.0, None)
    assert call(st=None) == 1
    assert call(N=-2) == 1
    assert call(dk=64) == 2
    assert call(dt=3) == 2
    assert call(st=MIS) == 3
    assert lib.kda_decode_step(F, F, F, F, ctypes.c_void_p(17), F, F, 0, 4, 2, 128, 128, 1.0, None) == 3


def test_workspace_sizes_are_queryable(lib):
    assert lib.kda_chunk_fwd_workspace_size(1, 8192, 32, 128, 128) >= 0
    assert lib.kda_varlen_fwd_workspace_size(4, 65536, 32, 128, 128) >= 0


def test_chunk_workspace_is_required_and_sized(lib):
    need = lib.kda_chunk_fwd_workspace_size(2, 100, 3, 128, 128)
    assert need == 2 * 2 * 3 * 66560 + 2 * 3 * 65536 + 256  # records, carried states, counter
    # valid shape, no workspace: rejected before anything is launched
    assert lib.kda_chunk_fwd(F, F, F, F, F, None, F, 1, None, 2, 100, 3, 128, 128, 1.0,
                             None, 0, None) == 7
    assert lib.kda_chunk_fwd(F, F, F, F, F, None, F, 1, None, 2, 100, 3, 128, 128, 1.0,
                             F, need - 16, None) == 7
    vneed = lib.kda_varlen_fwd_workspace_size(4, 1000, 2, 128, 128)
    assert vneed == 1024 + (1000 // 64 + 4) * 2 * 66560 + 4 * 2 * 65536 + 256


def test_checkpointed_argument_errors(lib):
    def call(every=512, ck=F, T=1024, ws=None, wsb=0):
        return lib.kda_chunk_fwd_checkpointed(F, F, F, F, F, None, F, 0, None, 1, T, 2, 128, 128,
                                              1.0, ck, every, ws, wsb, None)
    assert call(every=0) == 1             # not positive
    assert call(every=100) == 1           # not a multiple of 64
    assert call(ck=None) == 1             # checkpoints needed: T >= checkpoint_every
    assert call(ck=ctypes.c_void_p(24)) == 3
    assert call() == 7                    # valid, but no workspace


def test_speculative_argument_errors(lib):
    v = lambda N=2, K=3, dk=128, st=F, out=F: lib.kda_decode_verify(
        F, F, F, F, F, st, out, 1, N, K, 2, dk, 128, 1.0, None)
    assert v(N=-1) == 1
    assert v(dk=64) == 2
    assert v(st=ctypes.c_void_p(24)) == 3
    assert v(out=None) == 1
    assert v(N=0) == 0 and v(K=0) == 0
    c = lambda acc=F: lib.kda_decode_commit(F, F, F, F, F, F, acc, 2, 3, 2, 128, 128, None)
    assert c(acc=None) == 1


# The fixed-scratch entry point holds at most this many (chunk, head) records
# (the limit include/kda.h documents for kda_chunk_fwd_noalloc).
NOALLOC_MAX_RECORDS = 1008


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    call = lambda B, T, H: lib.kda_chunk_fwd_noalloc(F, F, F, F, F, None, F, 1, None, B, T, H,
                                                     128, 128, 1.0, None)
    # 1 * ceil(4096 / 64) * 32 = 2048 records: refused before any launch
    assert call(1, 4096, 32) == 7
    # one record over the limit
    assert call(1, 64 * (NOALLOC_MAX_RECORDS + 1), 1) == 7
    assert call(-1, 64, 1) == 1
