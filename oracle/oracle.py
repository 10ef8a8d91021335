"""KDA forward oracle -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this module.  It shares
no code with the CUDA library and never imports it.

Three independent fp64 evaluations of the same layer:

* :func:`kda_recurrence` -- the token-by-token definition, in C (``kda_oracle.c``),
  threaded over (sequence, head, block of value columns).  This is the oracle.
* :func:`brute_force` -- dense transition matrices multiplied out, for T <= 8.
* :func:`segmented_forward` -- the sequence cut into segments, each reduced to a
  (cumulative transition, zero-start state) pair, composed by a prefix scan.
* :func:`chunked` -- the blockwise (chunked) algebra: intra-chunk pair decays,
  a triangular solve for the delta-rule corrections and a state hand-off
  between chunks.  It follows the chunked evaluation the orkas.ai page
  ("Kimi K3 architecture", section "Eine Untergrenze, die einen
  GPU-Codepfad beseitigte") says needs division by the accumulated decay,
  with every pair decay taken exactly as exp(g_r - g_i) instead.

The recurrence (the gated delta rule with one decay per key channel):

    S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,
    o_t = scale * S_t^T q_t,          alpha_t = exp(log_alpha_t).

The fixed-size, serially updated state is the one described in the orkas.ai
page, sections "Sequenz: Drei Viertel der Schichten lesen nicht mehr alles"
and "Die Rechnung landet in der Bereitstellungsinfrastruktur".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sysconfig

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libkda_oracle.so")
_lib = None

MUTATIONS = {
    "none": 0,
    "decay_after_write": 1,
    "output_before_write": 2,
    "drop_beta": 3,
    "sign": 4,
    "decay_on_columns": 5,
}


def build(force: bool = False) -> str:
    """Compile the C oracle (plain gcc, OpenMP, no fast-math)."""
    src = os.path.join(_HERE, "kda_oracle.c")
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= max(
        os.path.getmtime(src), os.path.getmtime(os.path.join(_HERE, "kda_oracle.h"))
    ):
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    cc = os.environ.get("CC", "gcc")
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(
        [cc, "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
         "-o", tmp, src, "-lm"]
    )
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        dp = ctypes.POINTER(ctypes.c_double)
        lib.kda_oracle_fwd.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.POINTER(ctypes.c_longlong), dp, dp, dp, dp, dp, dp,
            ctypes.c_double, dp, dp, ctypes.c_int, ctypes.c_int,
        ]
        lib.kda_oracle_fwd.restype = ctypes.c_int
        lib.kda_oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().kda_oracle_max_threads())


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):  # torch tensor -> exact fp64 copy on the host
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def kda_recurrence(q, k, v, log_alpha, beta, initial_state=None, scale=1.0,
                   cu_seqlens=None, threads=0, mutation="none"):
    """Token-by-token fp64 recurrence.

    Fixed length: q, k, log_alpha [B,T,H,dk]; v [B,T,H,dv]; beta [B,T,H];
    initial_state [B,H,dk,dv] or None.  Returns (out [B,T,H,dv], final [B,H,dk,dv]).

    Packed: pass cu_seqlens (N+1 ints) with tensors [T_total,H,*] (or with a
    leading 1); states are [N,H,dk,dv] and out is [T_total,H,dv].
    """
    q, k, v, log_alpha, beta = (_f64(x) for x in (q, k, v, log_alpha, beta))
    packed = cu_seqlens is not None
    if packed:
        if q.ndim == 4:
            q, k, v, log_alpha, beta = q[0], k[0], v[0], log_alpha[0], beta[0]
        T_total, H, dk = q.shape
        dv = v.shape[-1]
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
        N = len(cu) - 1
        if cu[0] != 0 or cu[-1] != T_total:
            raise ValueError("cu_seqlens must start at 0 and end at T_total")
    else:
        B, T, H, dk = q.shape
        dv = v.shape[-1]
        N = B
        cu = np.arange(B + 1, dtype=np.int64) * T
        q, k, v, log_alpha, beta = (x.reshape((B * T,) + x.shape[2:]) for x in
                                     (q, k, v, log_alpha, beta))
    q, k, v, log_alpha, beta = (np.ascontiguousarray(x) for x in (q, k, v, log_alpha, beta))
    s0 = None if initial_state is None else _f64(initial_state).reshape(N, H, dk, dv)
    out = np.zeros((q.shape[0], H, dv), dtype=np.float64)
    fin = np.zeros((N, H, dk, dv), dtype=np.float64)
    rc = _load().kda_oracle_fwd(
        N, H, dk, dv, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_longlong)),
        _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(s0),
        float(scale), _ptr(out), _ptr(fin), int(threads), MUTATIONS[mutation])
    if rc != 0:
        raise RuntimeError(f"kda_oracle_fwd failed with code {rc}")
    if not packed:
        out = out.reshape(N, -1, H, dv)
    return out, fin


def decode_step(q, k, v, log_alpha, beta, state, scale=1.0, threads=0):
    """One token per sequence: q,k,log_alpha [N,H,dk], v [N,H,dv], beta [N,H],
    state [N,H,dk,dv].  Returns (out [N,H,dv], new_state)."""
    q = _f64(q)
    N = q.shape[0]
    cu = np.arange(N + 1)
    return kda_recurrence(q, k, v, log_alpha, beta, state, scale, cu_seqlens=cu,
                          threads=threads)


def brute_force(q, k, v, log_alpha, beta, initial_state=None, scale=1.0):
    """Dense transitions multiplied out, for one sequence of T <= 8 tokens.

    M_t = (I - beta_t k_t k_t^T) Diag(alpha_t);  S_t = M_t...M_1 S_0 +
    sum_{s<=t} M_t...M_{s+1} beta_s k_s v_s^T;  o_t = scale S_t^T q_t.
    Inputs [T,H,d]; every S_t is rebuilt from the products, never updated.
    """
    q, k, v, log_alpha, beta = (_f64(x) for x in (q, k, v, log_alpha, beta))
    T, H, dk = q.shape
    dv = v.shape[-1]
    if T > 8:
        raise ValueError("brute force is meant for T <= 8")
    s0 = np.zeros((H, dk, dv)) if initial_state is None else _f64(initial_state).reshape(H, dk, dv)
    out = np.zeros((T, H, dv))
    fin = np.zeros((H, dk, dv))
    eye = np.eye(dk)
    for h in range(H):
        M = [(eye - beta[t, h] * np.outer(k[t, h], k[t, h])) @ np.diag(np.exp(log_alpha[t, h]))
             for t in range(T)]
        for t in range(T):
            P = eye.copy()
            for s in range(t + 1):
                P = M[s] @ P
            S = P @ s0[h]
            for s in range(t + 1):
                R = eye.copy()
                for m in range(s + 1, t + 1):
                    R = M[m] @ R
                S = S + R @ (beta[s, h] * np.outer(k[s, h], v[s, h]))
            out[t, h] = scale * (S.T @ q[t, h])
            if t == T - 1:
                fin[h] = S
    if T == 0:
        fin = s0.copy()
    return out, fin


def _forward_substitution(L, B):
    """Solve L X = B for unit lower-triangular L, row by row."""
    X = np.zeros_like(B)
    for r in range(L.shape[0]):
        X[r] = B[r] - L[r, :r] @ X[:r]
    return X


def chunked(q, k, v, log_alpha, beta, initial_state=None, scale=1.0, chunk=64):
    """Blockwise evaluation of one sequence ([T,H,d] inputs) in fp64.

    Within a chunk, with g the inclusive cumulative log-decay from the chunk
    start and S_0 the state entering the chunk:
      A_kk[r,i] = beta_r sum_c k_rc k_ic exp(g_rc - g_ic)   (i < r)
      A_qk[r,i] = sum_c q_rc k_ic exp(g_rc - g_ic)           (i <= r)
      (I + A_kk) U = diag(beta) (V - (k * exp(g)) S_0)        forward substitution
      O   = (q * exp(g)) S_0 + A_qk U
      S_C = Diag(exp(g_C)) S_0 + (k * exp(g_C - g))^T U
    The pair decays exp(g_r - g_i) are evaluated directly for i <= r.
    """
    q, k, v, log_alpha, beta = (_f64(x) for x in (q, k, v, log_alpha, beta))
    T, H, dk = q.shape
    dv = v.shape[-1]
    S = np.zeros((H, dk, dv)) if initial_state is None else _f64(initial_state).reshape(H, dk, dv).copy()
    out = np.zeros((T, H, dv))
    for h in range(H):
        for t0 in range(0, T, chunk):
            t1 = min(T, t0 + chunk)
            C = t1 - t0
            qc, kc, vc = q[t0:t1, h], k[t0:t1, h], v[t0:t1, h]
            bc = beta[t0:t1, h]
            g = np.cumsum(log_alpha[t0:t1, h], axis=0)           # [C, dk]
            diff = g[:, None, :] - g[None, :, :]                    # [r, i, c]
            lower = np.tril(np.ones((C, C), dtype=bool))           # i <= r
            decay = np.where(lower[:, :, None], np.exp(np.where(lower[:, :, None], diff, 0.0)), 0.0)
            A_qk = np.einsum("rc,ic,ric->ri", qc, kc, decay)
            A_kk = bc[:, None] * np.einsum("rc,ic,ric->ri", kc, kc, decay)
            A_kk = np.tril(A_kk, -1)
            rhs = bc[:, None] * (vc - (kc * np.exp(g)) @ S[h])
            U = _forward_substitution(np.eye(C) + A_kk, rhs)
            out[t0:t1, h] = scale * ((qc * np.exp(g)) @ S[h] + A_qk @ U)
            S[h] = np.exp(g[-1])[:, None] * S[h] + (kc * np.exp(g[-1][None, :] - g)).T @ U
    return out, S


# ---------------------------------------------------------------------------
# Sequence split into segments (context parallelism).  The orkas.ai page
# ("Kimi K3 architecture", section "Die Rechnung landet in der
# Bereitstellungsinfrastruktur") explains why per-segment states cannot just
# be added for KDA: every token applies a transition to the state it
# receives.  Each segment is therefore reduced to two quantities that
# compose, its cumulative transition and the state it produces from a zero
# start, and every segment's entry state is rebuilt by a prefix scan over
# those pairs.  Written here for one sequence ([T, H, d] inputs), in fp64.
#
#   S_out = M S_in + Z          (M: [d_k, d_k], Z: [d_k, d_v], per head)
#   M = prod_t (I - beta_t k_t k_t^T) Diag(alpha_t)     (latest token leftmost)
#   Z = the segment's final state from S_in = 0
#   (M1, Z1) then (M2, Z2)  ->  (M2 M1, M2 Z1 + Z2)


def segment_transition(k, log_alpha, beta):
    """Cumulative transition M [H, dk, dk] of one segment ([T, H, dk] k and
    log_alpha, [T, H] beta), applying the tokens' transitions in order."""
    k, log_alpha, beta = (_f64(x) for x in (k, log_alpha, beta))
    T, H, dk = k.shape
    M = np.broadcast_to(np.eye(dk), (H, dk, dk)).copy()
    for t in range(T):
        M = np.exp(log_alpha[t])[:, :, None] * M                       # Diag(alpha_t) M
        M -= beta[t][:, None, None] * k[t][:, :, None] * np.einsum("hc,hcj->hj", k[t], M)[:, None, :]
    return M


def segment_summary(k, v, log_alpha, beta):
    """(M, Z) of one segment ([T, H, *] inputs): its cumulative transition and
    its final state from a zero entering state (the token-by-token recurrence)."""
    k, v, log_alpha, beta = (_f64(x) for x in (k, v, log_alpha, beta))
    _, Z = kda_recurrence(np.zeros_like(k)[None], k[None], v[None], log_alpha[None], beta[None])
    return segment_transition(k, log_alpha, beta), Z[0]


def compose_summaries(first, second):
    """The pair of two consecutive segments, `first` then `second`."""
    (M1, Z1), (M2, Z2) = first, second
    return M2 @ M1, M2 @ Z1 + Z2


def segment_entry_states(summaries, initial_state):
    """Exclusive prefix scan: the state entering each segment, and the final
    state after the last."""
    S = _f64(initial_state).copy()
    entries = []
    for M, Z in summaries:
        entries.append(S)
        S = M @ S + Z
    return entries, S


def segmented_forward(q, k, v, log_alpha, beta, initial_state=None, scale=1.0, seg_len=64):
    """The layer over one sequence split into segments of seg_len tokens: each
    segment's (M, Z) pair independently, the prefix scan for the entry states,
    then each segment again from its entry state.  Returns (out [T, H, dv],
    final [H, dk, dv]); equal to kda_recurrence up to rounding."""
    q, k, v, log_alpha, beta = (_f64(x) for x in (q, k, v, log_alpha, beta))
    T, H, dk = q.shape
    dv = v.shape[-1]
    S0 = np.zeros((H, dk, dv)) if initial_state is None else _f64(initial_state).reshape(H, dk, dv)
    bounds = [(t0, min(T, t0 + seg_len)) for t0 in range(0, T, seg_len)]
    summaries = [segment_summary(k[a:b], v[a:b], log_alpha[a:b], beta[a:b]) for a, b in bounds]
    entries, final = segment_entry_states(summaries, S0)
    out = np.zeros((T, H, dv))
    for (a, b), E in zip(bounds, entries):
        o, _ = kda_recurrence(q[None, a:b], k[None, a:b], v[None, a:b], log_alpha[None, a:b],
                              beta[None, a:b], E[None], scale)
        out[a:b] = o[0]
    return out, final


# ---------------------------------------------------------------------------
# Backward pass (gradients of the layer), for training at 8k and then 64k
# contexts (the studioglobal.ai page, German edition, section "Große
# Kapazität ...").  The pages give no algorithm for it; this is the reverse
# of the token-by-token recurrence above, derived by hand, in fp64:
#
#   forward, per token:  S' = Diag(alpha) S_prev,   w = v - S'^T k,
#                        u = beta w,   S = S' + k u^T,   o = scale S^T q
#   backward, with G = dL/dS (starting from dL/dS_T) and do = dL/do:
#     G  += scale q do^T                    (o reads the updated state)
#     dq  = scale S do
#     du  = G^T k;     dk = G u;            dv = beta du;   dbeta = <du, w>
#     dS' = G - beta k du^T;     dk -= beta S' du
#     dalpha = rowsum(dS' * S_prev);        dlog_alpha = alpha * dalpha
#     G  <- Diag(alpha) dS'                 (the gradient of S_prev)
# after the first token, G is the gradient of the initial state.


def _loop_states(q, k, v, log_alpha, beta, S0):
    """Every state of one sequence: S[t] after token t (S[-1]... kept as S0)."""
    T, H, dk = k.shape
    states = np.zeros((T + 1,) + S0.shape)
    states[0] = S0
    for t in range(T):
        Sp = np.exp(log_alpha[t])[:, :, None] * states[t]
        u = beta[t][:, None] * (v[t] - np.einsum("hcv,hc->hv", Sp, k[t]))
        states[t + 1] = Sp + k[t][:, :, None] * u[:, None, :]
    return states


BWD_MUTATIONS = ("none", "carry_without_decay", "dk_without_correction", "output_after_update",
                 "dbeta_from_v")


def kda_recurrence_bwd(q, k, v, log_alpha, beta, initial_state, d_out, d_final=None,
                       scale=1.0, cu_seqlens=None, mutation="none"):
    """Gradients of L = <d_out, out> + <d_final, final_state> for the layer
    computed by kda_recurrence (same layouts; packed sequences with
    cu_seqlens).  Returns dict(q, k, v, log_alpha, beta, initial_state) of
    fp64 arrays shaped like the inputs (initial_state: [N, H, dk, dv]).
    `mutation` plants a known mistake for the tests that prove the pins catch
    it ("none" = the derivation above)."""
    if mutation not in BWD_MUTATIONS:
        raise ValueError(mutation)
    q, k, v, log_alpha, beta, d_out = (_f64(x) for x in (q, k, v, log_alpha, beta, d_out))
    packed = cu_seqlens is not None
    if packed:
        if q.ndim == 4:
            q, k, v, log_alpha, beta, d_out = (x[0] for x in (q, k, v, log_alpha, beta, d_out))
        cu = [int(c) for c in cu_seqlens]
    else:
        B, T = q.shape[:2]
        cu = [b * T for b in range(B + 1)]
        q, k, v, log_alpha, beta, d_out = (x.reshape((B * T,) + x.shape[2:]) for x in
                                           (q, k, v, log_alpha, beta, d_out))
    N = len(cu) - 1
    _, H, dk = q.shape
    dv = v.shape[-1]
    S0 = (np.zeros((N, H, dk, dv)) if initial_state is None
          else _f64(initial_state).reshape(N, H, dk, dv))
    dF = np.zeros((N, H, dk, dv)) if d_final is None else _f64(d_final).reshape(N, H, dk, dv)
    g = {name: np.zeros_like(x) for name, x in
         (("q", q), ("k", k), ("v", v), ("log_alpha", log_alpha), ("beta", beta))}
    g_s0 = np.zeros((N, H, dk, dv))
    for n in range(N):
        a, b = cu[n], cu[n + 1]
        states = _loop_states(q[a:b], k[a:b], v[a:b], log_alpha[a:b], beta[a:b], S0[n])
        G = dF[n].copy()
        for t in range(b - a - 1, -1, -1):
            tt = a + t
            alpha = np.exp(log_alpha[tt])                               # [H, dk]
            S_prev, S = states[t], states[t + 1]
            Sp = alpha[:, :, None] * S_prev
            w = v[tt] - np.einsum("hcv,hc->hv", Sp, k[tt])             # [H, dv]
            u = beta[tt][:, None] * w
            if mutation != "output_after_update":
                G = G + scale * q[tt][:, :, None] * d_out[tt][:, None, :]
            g["q"][tt] = scale * np.einsum("hcv,hv->hc", S, d_out[tt])
            du = np.einsum("hcv,hc->hv", G, k[tt])
            g["v"][tt] = beta[tt][:, None] * du
            g["beta"][tt] = np.einsum("hv,hv->h", du, v[tt] if mutation == "dbeta_from_v" else w)
            dSp = G - beta[tt][:, None, None] * k[tt][:, :, None] * du[:, None, :]
            g["k"][tt] = np.einsum("hcv,hv->hc", G, u)
            if mutation != "dk_without_correction":
                g["k"][tt] -= beta[tt][:, None] * np.einsum("hcv,hv->hc", Sp, du)
            g["log_alpha"][tt] = alpha * np.einsum("hcv,hcv->hc", dSp, S_prev)
            G = dSp if mutation == "carry_without_decay" else alpha[:, :, None] * dSp
            if mutation == "output_after_update":
                G = G + scale * q[tt][:, :, None] * d_out[tt][:, None, :]
        g_s0[n] = G
    if not packed:
        g = {name: x.reshape((B, T) + x.shape[1:]) for name, x in g.items()}
    g["initial_state"] = g_s0
    return g
