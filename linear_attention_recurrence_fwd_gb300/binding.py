"""ctypes binding over libkda.so.  Argument marshalling only: every step of
the layer runs in the library's kernels.  Torch supplies device memory and
the current stream; nothing here computes any part of the layer, and there
is no fallback when the library is missing -- the call raises.

The Python names match the C entry points (include/kda.h).
"""
from __future__ import annotations

import ctypes
import os

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libkda.so")
PROBE_LIB_PATH = os.path.join(PKG, "libkda_probe.so")

KDA_BF16, KDA_F32 = 0, 1
STATUS = {
    0: "ok", 1: "invalid argument", 2: "unsupported shape or dtype",
    3: "pointer not 16-byte aligned", 4: "CUDA error", 5: "log_alpha outside [-5, 0]",
    6: "device wait timed out", 7: "workspace too small",
    8: "state-pass operand outside the fp16 range",
}

EXPORTS = ["kda_chunk_fwd", "kda_chunk_fwd_workspace_size", "kda_chunk_fwd_noalloc",
           "kda_chunk_fwd_segments", "kda_chunk_fwd_segments_workspace_size",
           "kda_chunk_fwd_checkpointed", "kda_chunk_fwd_launches", "kda_decode_verify",
           "kda_chunk_bwd", "kda_chunk_bwd_workspace_size",
           "kda_chunk_fwd_host", "kda_chunk_fwd_host_workspace_size",
           "kda_decode_commit",
           "kda_varlen_fwd",
           "kda_varlen_fwd_workspace_size", "kda_decode_step", "kda_status_string",
           "kda_last_device_status", "kda_version"]


class KDAError(RuntimeError):
    def __init__(self, code, where):
        self.code = int(code)
        super().__init__(f"{where}: {STATUS.get(self.code, 'unknown')} (status {self.code})")


_lib = None
_probe = None

_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t


def load(path: str = LIB_PATH):
    """Load libkda.so (raises if it was not built: there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(
                f"libkda.so not found at {path}; build it with "
                "`python -m linear_attention_recurrence_fwd_gb300.build` (no CPU fallback exists)")
        lib = ctypes.CDLL(path)
        lib.kda_chunk_fwd.argtypes = [_vp] * 7 + [_i, _vp, _i, _i, _i, _i, _i, _f, _vp, _sz, _vp]
        lib.kda_chunk_fwd.restype = _i
        lib.kda_chunk_fwd_checkpointed.argtypes = ([_vp] * 7 + [_i, _vp, _i, _i, _i, _i, _i, _f] +
                                                   [_vp, _i, _vp, _sz, _vp])
        lib.kda_chunk_fwd_checkpointed.restype = _i
        lib.kda_chunk_fwd_host.argtypes = lib.kda_chunk_fwd.argtypes
        lib.kda_chunk_fwd_host.restype = _i
        lib.kda_chunk_fwd_host_workspace_size.argtypes = [_i] * 6
        lib.kda_chunk_fwd_host_workspace_size.restype = _sz
        lib.kda_chunk_bwd.argtypes = [_vp] * 14 + [_i, _i, _i, _i, _i, _f, _vp, _sz, _vp]
        lib.kda_chunk_bwd.restype = _i
        lib.kda_chunk_bwd_workspace_size.argtypes = [_i] * 5
        lib.kda_chunk_bwd_workspace_size.restype = _sz
        lib.kda_chunk_fwd_segments.argtypes = ([_vp] * 7 + [_i, _vp, _i, _i, _i, _i, _i, _f, _i] +
                                               [_vp, _sz, _vp])
        lib.kda_chunk_fwd_segments.restype = _i
        lib.kda_chunk_fwd_segments_workspace_size.argtypes = [_i] * 6
        lib.kda_chunk_fwd_segments_workspace_size.restype = _sz
        lib.kda_chunk_fwd_noalloc.argtypes = [_vp] * 7 + [_i, _vp, _i, _i, _i, _i, _i, _f, _vp]
        lib.kda_chunk_fwd_noalloc.restype = _i
        lib.kda_varlen_fwd.argtypes = [_vp] * 6 + [_i, _i, _i, _vp, _vp, _i, _vp, _i, _i, _i, _f,
                                                   _vp, _sz, _vp]
        lib.kda_varlen_fwd.restype = _i
        lib.kda_decode_step.argtypes = [_vp] * 7 + [_i, _i, _i, _i, _i, _f, _vp]
        lib.kda_decode_step.restype = _i
        lib.kda_decode_verify.argtypes = [_vp] * 7 + [_i, _i, _i, _i, _i, _i, _f, _vp]
        lib.kda_decode_verify.restype = _i
        lib.kda_decode_commit.argtypes = [_vp] * 7 + [_i, _i, _i, _i, _i, _vp]
        lib.kda_decode_commit.restype = _i
        lib.kda_chunk_fwd_workspace_size.argtypes = [_i] * 5
        lib.kda_chunk_fwd_workspace_size.restype = _sz
        lib.kda_varlen_fwd_workspace_size.argtypes = [_i] * 5
        lib.kda_varlen_fwd_workspace_size.restype = _sz
        lib.kda_chunk_fwd_launches.argtypes = [_i, _i, _i]
        lib.kda_chunk_fwd_launches.restype = _i
        lib.kda_status_string.argtypes = [_i]
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_last_device_status.argtypes = [_vp]
        lib.kda_last_device_status.restype = _i
        lib.kda_version.restype = ctypes.c_char_p
        _lib = lib
    return _lib


def load_probe(path: str = PROBE_LIB_PATH):
    """Test-only layout probes (libkda_probe.so)."""
    global _probe
    if _probe is None:
        if not os.path.exists(path):
            raise RuntimeError(f"libkda_probe.so not found at {path}")
        lib = ctypes.CDLL(path)
        lib.kda_probe_umma.argtypes = [_vp, _vp, _vp] + [_i] * 14 + [_vp, _vp]
        lib.kda_probe_umma.restype = _i
        lib.kda_probe_tma.argtypes = [_vp, _vp] + [_i] * 5 + [_vp, _vp]
        lib.kda_probe_tma.restype = _i
        lib.kda_probe_umma_ta.argtypes = [_vp, _vp, _vp] + [_i] * 15 + [_vp, _vp]
        lib.kda_probe_umma_ta.restype = _i
        lib.kda_probe_wait_timeout.argtypes = [_i, _vp, _vp]
        lib.kda_probe_wait_timeout.restype = _i
        _probe = lib
    return _probe


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(code, where):
    if code != 0:
        raise KDAError(code, where)


def _dtype_code(dt):
    if dt == torch.bfloat16:
        return KDA_BF16
    if dt == torch.float32:
        return KDA_F32
    raise ValueError(f"unsupported output dtype {dt}")


def _need(t, dtype, name):
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")


def _need_host(t, dtype, name):
    if t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous host {dtype} tensor")


def kda_chunk_fwd(q, k, v, log_alpha, beta, initial_state=None, scale=1.0,
                  out_dtype=torch.float32, output_final_state=True, out=None,
                  final_state=None, stream=None):
    """Chunked prefill.  q,k,log_alpha [B,T,H,dk] bf16; v [B,T,H,dv] bf16;
    beta [B,T,H] bf16; initial_state [B,H,dk,dv] fp32 or None.
    Returns (out [B,T,H,dv], final_state [B,H,dk,dv] fp32 or None)."""
    lib = load()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (log_alpha, "log_alpha"), (beta, "beta")):
        _need(t, torch.bfloat16, n)
    if initial_state is not None:
        _need(initial_state, torch.float32, "initial_state")
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=out_dtype, device=q.device)
    if final_state is None and output_final_state:
        final_state = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
    ws_bytes = lib.kda_chunk_fwd_workspace_size(B, T, H, dk, dv)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device) if ws_bytes else None
    _check(lib.kda_chunk_fwd(_p(q), _p(k), _p(v), _p(log_alpha), _p(beta), _p(initial_state),
                             _p(out), _dtype_code(out.dtype), _p(final_state), B, T, H, dk, dv,
                             float(scale), _p(ws), ws_bytes, _stream(stream)), "kda_chunk_fwd")
    return out, final_state


def kda_chunk_fwd_segments(q, k, v, log_alpha, beta, initial_state=None, scale=1.0,
                           n_segments=2, out_dtype=torch.float32, out=None, final_state=None,
                           stream=None):
    """kda_chunk_fwd with each sequence cut into n_segments segments walked in
    parallel and joined by a scan of their (transition, zero-start state)
    pairs.  Returns (out, final_state)."""
    lib = load()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (log_alpha, "log_alpha"), (beta, "beta")):
        _need(t, torch.bfloat16, n)
    if initial_state is not None:
        _need(initial_state, torch.float32, "initial_state")
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=out_dtype, device=q.device)
    if final_state is None:
        final_state = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
    ws_bytes = lib.kda_chunk_fwd_segments_workspace_size(B, T, H, dk, dv, int(n_segments))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device) if ws_bytes else None
    _check(lib.kda_chunk_fwd_segments(
        _p(q), _p(k), _p(v), _p(log_alpha), _p(beta), _p(initial_state), _p(out),
        _dtype_code(out.dtype), _p(final_state), B, T, H, dk, dv, float(scale), int(n_segments),
        _p(ws), ws_bytes, _stream(stream)), "kda_chunk_fwd_segments")
    return out, final_state


def kda_chunk_fwd_checkpointed(q, k, v, log_alpha, beta, initial_state=None, scale=1.0,
                               checkpoint_every=512, out_dtype=torch.float32, out=None,
                               final_state=None, checkpoints=None, stream=None):
    """kda_chunk_fwd plus the state after every `checkpoint_every` tokens.
    Returns (out, final_state, checkpoints [B, T // checkpoint_every, H, dk, dv])."""
    lib = load()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (log_alpha, "log_alpha"), (beta, "beta")):
        _need(t, torch.bfloat16, n)
    if initial_state is not None:
        _need(initial_state, torch.float32, "initial_state")
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=out_dtype, device=q.device)
    if final_state is None:
        final_state = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
    n_ckpt = T // checkpoint_every if checkpoint_every > 0 else 0
    if checkpoints is None:
        checkpoints = torch.empty((B, n_ckpt, H, dk, dv), dtype=torch.float32, device=q.device)
    ws_bytes = lib.kda_chunk_fwd_workspace_size(B, T, H, dk, dv)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device) if ws_bytes else None
    _check(lib.kda_chunk_fwd_checkpointed(
        _p(q), _p(k), _p(v), _p(log_alpha), _p(beta), _p(initial_state), _p(out),
        _dtype_code(out.dtype), _p(final_state), B, T, H, dk, dv, float(scale),
        _p(checkpoints) if n_ckpt else None, int(checkpoint_every), _p(ws), ws_bytes,
        _stream(stream)), "kda_chunk_fwd_checkpointed")
    return out, final_state, checkpoints


def kda_chunk_fwd_host_workspace(B, T, H, dk=128, dv=128, out_dtype=torch.float32, device=None):
    """A device workspace for kda_chunk_fwd_host of this shape."""
    lib = load()
    n = lib.kda_chunk_fwd_host_workspace_size(B, T, H, dk, dv, _dtype_code(out_dtype))
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device or torch.device("cuda"))


def kda_chunk_fwd_host(q, k, v, log_alpha, beta, initial_state=None, scale=1.0,
                       out_dtype=torch.float32, out=None, final_state=None, workspace=None,
                       stream=None):
    """kda_chunk_fwd with every tensor in host memory (CPU tensors, ideally
    pinned): the library copies each round's inputs in and its outputs back
    while other rounds compute.  Returns (out, final_state) on the host."""
    lib = load()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (log_alpha, "log_alpha"), (beta, "beta")):
        _need_host(t, torch.bfloat16, n)
    if initial_state is not None:
        _need_host(initial_state, torch.float32, "initial_state")
    pin = q.is_pinned()
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=out_dtype, pin_memory=pin)
    if final_state is None:
        final_state = torch.empty((B, H, dk, dv), dtype=torch.float32, pin_memory=pin)
    if workspace is None:
        workspace = kda_chunk_fwd_host_workspace(B, T, H, dk, dv, out.dtype)
    _check(lib.kda_chunk_fwd_host(
        _p(q), _p(k), _p(v), _p(log_alpha), _p(beta), _p(initial_state), _p(out),
        _dtype_code(out.dtype), _p(final_state), B, T, H, dk, dv, float(scale), _p(workspace),
        workspace.numel(), _stream(stream)), "kda_chunk_fwd_host")
    return out, final_state


def kda_chunk_bwd(q, k, v, log_alpha, beta, d_out, initial_state=None, d_final_state=None,
                  scale=1.0, want_initial_state_grad=True, stream=None):
    """Gradients of <d_out, out> + <d_final_state, final_state> for the layer
    kda_chunk_fwd computes.  Returns a dict of fp32 tensors: q, k, v,
    log_alpha ([B, T, H, d]), beta ([B, T, H]) and initial_state
    ([B, H, dk, dv], or None when not asked for)."""
    lib = load()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (log_alpha, "log_alpha"), (beta, "beta")):
        _need(t, torch.bfloat16, n)
    _need(d_out, torch.float32, "d_out")
    for t, n in ((initial_state, "initial_state"), (d_final_state, "d_final_state")):
        if t is not None:
            _need(t, torch.float32, n)
    dev = q.device
    g = {name: torch.empty((B, T, H, d), dtype=torch.float32, device=dev)
         for name, d in (("q", dk), ("k", dk), ("v", dv), ("log_alpha", dk))}
    g["beta"] = torch.empty((B, T, H), dtype=torch.float32, device=dev)
    g["initial_state"] = (torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
                          if want_initial_state_grad else None)
    ws_bytes = lib.kda_chunk_bwd_workspace_size(B, T, H, dk, dv)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else None
    _check(lib.kda_chunk_bwd(
        _p(q), _p(k), _p(v), _p(log_alpha), _p(beta), _p(initial_state), _p(d_out),
        _p(d_final_state), _p(g["q"]), _p(g["k"]), _p(g["v"]), _p(g["log_alpha"]), _p(g["beta"]),
        _p(g["initial_state"]), B, T, H, dk, dv, float(scale), _p(ws), ws_bytes,
        _stream(stream)), "kda_chunk_bwd")
    return g


def kda_chunk_fwd_noalloc(q, k, v, log_alpha, beta, initial_state=None, scale=1.0,
                          out_dtype=torch.float32, output_final_state=True, out=None,
                          final_state=None, stream=None):
    """kda_chunk_fwd without a workspace: the library's fixed device scratch is
    used instead (B * ceil(T/64) * H <= 1008).  Outputs are allocated here
    only when not passed in; pass `out` / `final_state` to allocate nothing."""
    lib = load()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (log_alpha, "log_alpha"), (beta, "beta")):
        _need(t, torch.bfloat16, n)
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=out_dtype, device=q.device)
    if final_state is None and output_final_state:
        final_state = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
    _check(lib.kda_chunk_fwd_noalloc(_p(q), _p(k), _p(v), _p(log_alpha), _p(beta),
                                     _p(initial_state), _p(out), _dtype_code(out.dtype),
                                     _p(final_state), B, T, H, dk, dv, float(scale),
                                     _stream(stream)), "kda_chunk_fwd_noalloc")
    return out, final_state


def kda_varlen_fwd(q, k, v, log_alpha, beta, cu_seqlens, max_seqlen, initial_state=None,
                   scale=1.0, out_dtype=torch.float32, output_final_state=True, out=None,
                   final_state=None, stream=None):
    """Packed prefill.  Tensors [T_total,H,*] (or [1,T_total,H,*]);
    cu_seqlens int32 [N+1] on the device.  Returns (out, final_state [N,H,dk,dv])."""
    lib = load()
    squeeze = q.dim() == 4
    if squeeze:
        q, k, v, log_alpha, beta = q[0], k[0], v[0], log_alpha[0], beta[0]
    T_total, H, dk = q.shape
    dv = v.shape[-1]
    N = cu_seqlens.numel() - 1
    _need(cu_seqlens, torch.int32, "cu_seqlens")
    if out is None:
        out = torch.empty((T_total, H, dv), dtype=out_dtype, device=q.device)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, dk, dv), dtype=torch.float32, device=q.device)
    ws_bytes = lib.kda_varlen_fwd_workspace_size(N, T_total, H, dk, dv)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device) if ws_bytes else None
    _check(lib.kda_varlen_fwd(_p(q), _p(k), _p(v), _p(log_alpha), _p(beta), _p(cu_seqlens), N,
                              T_total, int(max_seqlen), _p(initial_state), _p(out),
                              _dtype_code(out.dtype), _p(final_state), H, dk, dv, float(scale),
                              _p(ws), ws_bytes, _stream(stream)), "kda_varlen_fwd")
    return (out[None] if squeeze else out), final_state


def kda_decode_step(q, k, v, log_alpha, beta, state, scale=1.0, out=None,
                    out_dtype=torch.float32, stream=None):
    """One token per sequence; `state` [N,H,dk,dv] fp32 is updated in place.
    q,k,log_alpha [N,H,dk], v [N,H,dv], beta [N,H] (bf16).  Returns out [N,H,dv]."""
    lib = load()
    N, H, dk = q.shape
    dv = v.shape[-1]
    _need(state, torch.float32, "state")
    if out is None:
        out = torch.empty((N, H, dv), dtype=out_dtype, device=q.device)
    _check(lib.kda_decode_step(_p(q), _p(k), _p(v), _p(log_alpha), _p(beta), _p(state), _p(out),
                               _dtype_code(out.dtype), N, H, dk, dv, float(scale),
                               _stream(stream)), "kda_decode_step")
    return out


def kda_decode_verify(q, k, v, log_alpha, beta, state, scale=1.0, out_dtype=torch.float32,
                      out=None, stream=None):
    """Outputs of K drafted tokens per sequence from `state` (only read).
    q, k, log_alpha, v [N,K,H,d] bf16; beta [N,K,H]; state [N,H,d,d] fp32.
    Returns out [N,K,H,d]."""
    lib = load()
    N, K, H, dk = q.shape
    dv = v.shape[-1]
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (log_alpha, "log_alpha"), (beta, "beta")):
        _need(t, torch.bfloat16, n)
    _need(state, torch.float32, "state")
    if out is None:
        out = torch.empty((N, K, H, dv), dtype=out_dtype, device=q.device)
    _check(lib.kda_decode_verify(_p(q), _p(k), _p(v), _p(log_alpha), _p(beta), _p(state),
                                 _p(out), _dtype_code(out.dtype), N, K, H, dk, dv, float(scale),
                                 _stream(stream)), "kda_decode_verify")
    return out


def kda_decode_commit(q, k, v, log_alpha, beta, state, accepted, stream=None):
    """Advance `state` in place by the first accepted[n] draft tokens of each
    sequence (accepted: int32 [N] on the device)."""
    lib = load()
    N, K, H, dk = q.shape
    dv = v.shape[-1]
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (log_alpha, "log_alpha"), (beta, "beta")):
        _need(t, torch.bfloat16, n)
    _need(state, torch.float32, "state")
    _need(accepted, torch.int32, "accepted")
    _check(lib.kda_decode_commit(_p(q), _p(k), _p(v), _p(log_alpha), _p(beta), _p(state),
                                 _p(accepted), N, K, H, dk, dv, _stream(stream)),
           "kda_decode_commit")
    return state


def kda_chunk_fwd_launches(B, T, H):
    """Kernel launches one kda_chunk_fwd call of this shape makes on the current device."""
    return int(load().kda_chunk_fwd_launches(int(B), int(T), int(H)))


def kda_last_device_status(stream=None) -> int:
    return int(load().kda_last_device_status(_stream(stream)))


def kda_status_string(code: int) -> str:
    return load().kda_status_string(int(code)).decode()


def kda_version() -> str:
    return load().kda_version().decode()
