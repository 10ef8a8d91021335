"""Pins for the fp64 oracle: each checks it against something other than
itself -- dense products, the chunked algebra, closed forms, invariants and
the constants the pages print.  CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from linear_attention_recurrence_fwd_gb300 import inputs as gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(T, H, dk, dv, seed, decay_mean=0.0, init=True, unit_keys=True):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    if unit_keys:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    beta = 1 / (1 + np.exp(-rng.standard_normal((T, H))))
    la = -5 / (1 + np.exp(-(rng.standard_normal((T, H, dk)) + decay_mean)))
    s0 = rng.standard_normal((H, dk, dv)) * 0.5 if init else None
    return q, k, v, la, beta, s0


def _run(q, k, v, la, beta, s0=None, scale=1.0, mutation="none"):
    out, fin = orc.kda_recurrence(q[None], k[None], v[None], la[None], beta[None],
                                  None if s0 is None else s0[None], scale=scale,
                                  mutation=mutation)
    return out[0], fin[0]


def _rel(a, b):
    return np.abs(a - b).max() / max(np.abs(b).max(), 1e-300)


@pytest.mark.parametrize("T,H,dk,dv", [(1, 1, 3, 2), (5, 2, 4, 3), (8, 2, 6, 5), (7, 1, 9, 9)])
def test_brute_force_products(T, H, dk, dv):
    q, k, v, la, beta, s0 = _rand(T, H, dk, dv, seed=T * 100 + dk)
    o, s = _run(q, k, v, la, beta, s0, scale=0.7)
    ob, sb = orc.brute_force(q, k, v, la, beta, s0, scale=0.7)
    assert _rel(o, ob) < 1e-12
    assert _rel(s, sb) < 1e-12


@pytest.mark.parametrize("chunk", [1, 16, 64, 150])
@pytest.mark.parametrize("decay_mean", [0.0, 2.0])
def test_chunked_reformulation(chunk, decay_mean):
    q, k, v, la, beta, s0 = _rand(150, 2, 16, 8, seed=7, decay_mean=decay_mean)
    o, s = _run(q, k, v, la, beta, s0)
    oc, sc = orc.chunked(q, k, v, la, beta, s0, chunk=chunk)
    assert _rel(o, oc) < 1e-10
    assert _rel(s, sc) < 1e-10


def test_chunked_slow_decay_long_memory():
    # state survives many chunks: the inter-chunk hand-off is really exercised
    q, k, v, la, beta, s0 = _rand(300, 1, 8, 4, seed=3)
    la = la * 0.01
    o, s = _run(q, k, v, la, beta, s0)
    oc, sc = orc.chunked(q, k, v, la, beta, s0, chunk=64)
    assert _rel(o, oc) < 1e-10 and _rel(s, sc) < 1e-10


def test_pure_decay_when_beta_zero():
    q, k, v, la, beta, s0 = _rand(40, 2, 6, 5, seed=11)
    beta[:] = 0.0
    o, s = _run(q, k, v, la, beta, s0)
    g = np.cumsum(la, axis=0)  # [T,H,dk]
    expect_s = np.exp(g[-1])[:, :, None] * s0
    assert _rel(s, expect_s) < 1e-13
    for t in range(40):
        st = np.exp(g[t])[:, :, None] * s0
        np.testing.assert_allclose(o[t], np.einsum("hcj,hc->hj", st, q[t]), rtol=1e-12, atol=1e-14)


def test_identity_when_no_decay_and_no_write():
    q, k, v, la, beta, s0 = _rand(33, 2, 5, 7, seed=12)
    la[:] = 0.0
    beta[:] = 0.0
    o, s = _run(q, k, v, la, beta, s0)
    assert np.array_equal(s, s0)  # bit-exact: exp(0) = 1, beta = 0


def test_delta_write_recalls_value():
    # beta = 1, unit keys: right after the write, S_t^T k_t = v_t
    q, k, v, la, beta, s0 = _rand(6, 1, 8, 4, seed=13)
    beta[:] = 1.0
    for t in range(1, 7):
        _, s = _run(q[:t], k[:t], v[:t], la[:t], beta[:t], s0)
        np.testing.assert_allclose(s[0].T @ k[t - 1, 0], v[t - 1, 0], atol=1e-12)


def test_orthonormal_keys_reduce_to_causal_linear_attention():
    # no decay, keys from an orthonormal basis, zero start: the delta rule
    # never corrects, so S_t = sum_s beta_s k_s v_s^T and the output is causal
    # (masked) linear attention with beta-weighted values.
    T, dk, dv = 12, 16, 5
    rng = np.random.default_rng(5)
    basis, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    k = basis[:, :T].T[:, None, :]          # [T,1,dk], mutually orthonormal
    q = rng.standard_normal((T, 1, dk))
    v = rng.standard_normal((T, 1, dv))
    beta = rng.uniform(0.1, 1.0, (T, 1))
    la = np.zeros((T, 1, dk))
    o, s = _run(q, k, v, la, beta)
    scores = np.tril(q[:, 0] @ k[:, 0].T) * beta[:, 0][None, :]
    np.testing.assert_allclose(o[:, 0], scores @ v[:, 0], atol=1e-12)
    np.testing.assert_allclose(s[0], (beta[:, 0, None] * k[:, 0]).T @ v[:, 0], atol=1e-12)


def test_scalar_case_geometric_series():
    # d_k = d_v = 1, constant coefficients: s_t = a s_{t-1} + b with
    # a = (1 - beta k^2) alpha, b = beta k v, so s_T = a^T s_0 + b (1-a^T)/(1-a)
    T = 50
    kk, vv, bb, al, s0v, qq = 0.8, -1.3, 0.6, 0.9, 0.4, 1.7
    q = np.full((T, 1, 1), qq)
    k = np.full((T, 1, 1), kk)
    v = np.full((T, 1, 1), vv)
    beta = np.full((T, 1), bb)
    la = np.full((T, 1, 1), math.log(al))
    o, s = _run(q, k, v, la, beta, np.full((1, 1, 1), s0v))
    a = (1 - bb * kk * kk) * al
    b = bb * kk * vv
    for t in range(1, T + 1):
        st = a ** t * s0v + b * (1 - a ** t) / (1 - a)
        assert abs(o[t - 1, 0, 0] - qq * st) < 1e-13
    assert abs(s[0, 0, 0] - (a ** T * s0v + b * (1 - a ** T) / (1 - a))) < 1e-13


def test_linearity_in_state_and_values():
    q, k, v, la, beta, s0 = _rand(70, 2, 6, 4, seed=21)
    o, s = _run(q, k, v, la, beta, s0)
    o1, s1 = _run(q, k, v, la, beta, s0 * 0.0 + s0)
    o2, s2 = _run(q, k, np.zeros_like(v), la, beta, s0)
    o3, s3 = _run(q, k, v, la, beta, np.zeros_like(s0))
    np.testing.assert_allclose(o, o2 + o3, atol=1e-12)
    np.testing.assert_allclose(s, s2 + s3, atol=1e-12)
    o4, s4 = _run(q, k, 2.5 * v, la, beta, 2.5 * s0)
    np.testing.assert_allclose(o4, 2.5 * o, atol=1e-12)


def test_heads_and_columns_independent():
    q, k, v, la, beta, s0 = _rand(40, 3, 6, 8, seed=22)
    o, s = _run(q, k, v, la, beta, s0)
    perm = [2, 0, 1]
    op, sp = _run(q[:, perm], k[:, perm], v[:, perm], la[:, perm], beta[:, perm], s0[perm])
    assert np.array_equal(op, o[:, perm]) and np.array_equal(sp, s[perm])
    # value columns split in two halves
    oa, sa = _run(q, k, v[..., :3], la, beta, s0[..., :3])
    ob, sb = _run(q, k, v[..., 3:], la, beta, s0[..., 3:])
    np.testing.assert_allclose(np.concatenate([oa, ob], -1), o, atol=1e-14)
    np.testing.assert_allclose(np.concatenate([sa, sb], -1), s, atol=1e-14)


@pytest.mark.parametrize("T1", [1, 37, 64, 100])
def test_split_and_resume(T1):
    q, k, v, la, beta, s0 = _rand(130, 2, 8, 6, seed=23)
    o, s = _run(q, k, v, la, beta, s0)
    oa, sa = _run(q[:T1], k[:T1], v[:T1], la[:T1], beta[:T1], s0)
    ob, sb = _run(q[T1:], k[T1:], v[T1:], la[T1:], beta[T1:], sa)
    np.testing.assert_allclose(np.concatenate([oa, ob]), o, atol=1e-13)
    np.testing.assert_allclose(sb, s, atol=1e-13)


def test_packed_sequences_equal_separate_runs():
    lens = [5, 64, 1, 90]
    H, dk, dv = 2, 8, 4
    parts = [_rand(n, H, dk, dv, seed=30 + i) for i, n in enumerate(lens)]
    cat = lambda j: np.concatenate([p[j] for p in parts])
    s0 = np.stack([p[5] for p in parts])
    cu = np.concatenate([[0], np.cumsum(lens)])
    o, s = orc.kda_recurrence(cat(0), cat(1), cat(2), cat(3), cat(4), s0, cu_seqlens=cu)
    for i, p in enumerate(parts):
        oi, si = _run(*p[:5], p[5])
        assert np.array_equal(o[cu[i]:cu[i + 1]], oi)
        assert np.array_equal(s[i], si)


def test_decode_step_is_one_token_of_the_recurrence():
    q, k, v, la, beta, s0 = _rand(1, 4, 8, 8, seed=40)
    # 4 "sequences" of one token each, H = 1
    o, s = orc.decode_step(q[:, :, None][0], k[:, :, None][0], v[:, :, None][0],
                           la[:, :, None][0], beta[0][:, None], s0[:, None])
    for n in range(4):
        on, sn = _run(q[:, n:n + 1], k[:, n:n + 1], v[:, n:n + 1], la[:, n:n + 1],
                      beta[:, n:n + 1], s0[n:n + 1])
        np.testing.assert_allclose(o[n, 0], on[0, 0], atol=0)
        np.testing.assert_allclose(s[n, 0], sn[0], atol=0)


def test_threads_do_not_change_results():
    q, k, v, la, beta, s0 = _rand(64, 3, 16, 24, seed=41)
    o1, s1 = orc.kda_recurrence(q[None], k[None], v[None], la[None], beta[None], s0[None], threads=1)
    o4, s4 = orc.kda_recurrence(q[None], k[None], v[None], la[None], beta[None], s0[None], threads=4)
    assert np.array_equal(o1, o4) and np.array_equal(s1, s4)


@pytest.mark.parametrize("mutation", ["decay_after_write", "output_before_write", "drop_beta",
                                      "sign", "decay_on_columns"])
def test_planted_mistakes_are_caught(mutation):
    """Each planted mistake must break at least one pin (here: the dense
    products), so the pins above have teeth."""
    q, k, v, la, beta, s0 = _rand(6, 2, 5, 5, seed=50)
    o, s = _run(q, k, v, la, beta, s0, mutation=mutation)
    ob, sb = orc.brute_force(q, k, v, la, beta, s0)
    assert max(_rel(o, ob), _rel(s, sb)) > 1e-3


def test_decay_bound_constants_from_the_page():
    g = json.load(open(os.path.join(GOLDEN, "decay_bound.json")))
    # 0.67 % kept per step  <=>  log_alpha >= -5
    assert round(math.exp(-5), 4) == g["min_kept_fraction_per_step"]
    lo, hi = g["tile_cumulative_logdecay_interval"]
    assert g["tile_tokens"] * -5 == lo and hi == 0
    # reciprocal of the tile decay e^80 ~ 5.5e34, inside the bf16 range ~3.4e38
    assert float(f"{math.exp(80):.1e}") == g["reciprocal_bound"]
    bf16_max = torch.finfo(torch.bfloat16).max
    assert float(f"{bf16_max:.1e}") == g["bf16_range"]
    assert math.exp(80) < bf16_max and math.exp(80) < torch.finfo(torch.float32).max


@pytest.mark.parametrize("name", ["tiny", "prefill_8k"])
def test_generated_inputs_respect_the_bound(name):
    w = gen.WORKLOADS[name]
    x = gen.workload_inputs(w, T=min(w.T, 2048))
    la = x["log_alpha"].float()
    assert la.min().item() >= -5.0 and la.max().item() <= 0.0
    T = la.shape[1] // 16 * 16
    tiles = la[:, :T].reshape(la.shape[0], T // 16, 16, *la.shape[2:]).double().sum(2)
    assert tiles.min().item() >= -80.0
    kn = x["k"].float().norm(dim=-1)
    assert (kn - 1).abs().max().item() < 2 ** -6
    b = x["beta"].float()
    assert b.min().item() > 0 and b.max().item() < 1
