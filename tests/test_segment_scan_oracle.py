"""Pins for the oracle's segment split (the orkas.ai page, "Kimi K3
architecture", section "Die Rechnung landet in der
Bereitstellungsinfrastruktur"): each segment reduces to a cumulative
transition M and a zero-start state Z, the pairs compose, and a prefix scan
over them gives every segment's entry state.  Checked against the
token-by-token recurrence, closed forms and the composition algebra."""
import numpy as np
import pytest

from oracle import oracle as orc


def _inputs(T, H, d, seed, decay=0.5):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, H, d))
    k = rng.standard_normal((T, H, d))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, d))
    la = -rng.uniform(0.0, decay, (T, H, d))
    beta = rng.uniform(0.0, 1.0, (T, H))
    S0 = rng.standard_normal((H, d, d))
    return q, k, v, la, beta, S0


@pytest.mark.parametrize("T,seg", [(150, 37), (150, 1), (150, 150), (128, 64), (65, 64)])
def test_segmented_forward_equals_token_loop(T, seg):
    q, k, v, la, beta, S0 = _inputs(T, 2, 16, seed=T + seg)
    ro, rs = orc.kda_recurrence(q[None], k[None], v[None], la[None], beta[None], S0[None], 0.7)
    so, ss = orc.segmented_forward(q, k, v, la, beta, S0, 0.7, seg_len=seg)
    assert np.abs(so - ro[0]).max() <= 1e-12 * max(1.0, np.abs(ro).max())
    assert np.abs(ss - rs[0]).max() <= 1e-12 * max(1.0, np.abs(rs).max())


def test_segment_state_is_affine_in_the_entering_state():
    """The recurrence's final state from any S_in is M S_in + Z."""
    q, k, v, la, beta, S0 = _inputs(40, 2, 12, seed=5)
    M, Z = orc.segment_summary(k, v, la, beta)
    for S_in in (S0, 3.0 * S0[:, ::-1]):
        _, fin = orc.kda_recurrence(q[None], k[None], v[None], la[None], beta[None], S_in[None])
        assert np.allclose(fin[0], M @ S_in + Z, rtol=1e-12, atol=1e-12)


def test_pure_decay_transition_is_diagonal():
    """beta = 0: no writes, M = Diag(exp(sum log_alpha)), Z = 0."""
    q, k, v, la, _, _ = _inputs(30, 2, 8, seed=6)
    beta = np.zeros((30, 2))
    M, Z = orc.segment_summary(k, v, la, beta)
    for h in range(2):
        assert np.allclose(M[h], np.diag(np.exp(la[:, h].sum(0))), rtol=1e-12, atol=1e-14)
    assert np.abs(Z).max() == 0.0


def test_single_token_transition():
    q, k, v, la, beta, _ = _inputs(1, 1, 6, seed=7)
    M = orc.segment_transition(k, la, beta)[0]
    kk, a, b = k[0, 0], np.exp(la[0, 0]), beta[0, 0]
    assert np.allclose(M, (np.eye(6) - b * np.outer(kk, kk)) @ np.diag(a), rtol=1e-13, atol=1e-14)


def test_pairs_compose_and_composition_is_associative():
    q, k, v, la, beta, _ = _inputs(90, 2, 10, seed=8)
    parts = [(0, 25), (25, 60), (60, 90)]
    s = [orc.segment_summary(k[a:b], v[a:b], la[a:b], beta[a:b]) for a, b in parts]
    whole = orc.segment_summary(k, v, la, beta)
    left = orc.compose_summaries(orc.compose_summaries(s[0], s[1]), s[2])
    right = orc.compose_summaries(s[0], orc.compose_summaries(s[1], s[2]))
    for got in (left, right):
        assert np.allclose(got[0], whole[0], rtol=1e-12, atol=1e-13)
        assert np.allclose(got[1], whole[1], rtol=1e-12, atol=1e-13)


def test_adding_zero_start_states_is_not_the_answer():
    """The page's point: summing the segments' zero-start states, as plain
    linear attention may, misses the transitions applied to the incoming state."""
    q, k, v, la, beta, _ = _inputs(120, 1, 8, seed=9)
    s = [orc.segment_summary(k[a:a + 40], v[a:a + 40], la[a:a + 40], beta[a:a + 40])
         for a in (0, 40, 80)]
    _, fin = orc.kda_recurrence(q[None], k[None], v[None], la[None], beta[None])
    naive = sum(Z for _, Z in s)
    _, scanned = orc.segment_entry_states(s, np.zeros_like(fin[0]))
    assert np.allclose(scanned, fin[0], rtol=1e-12, atol=1e-13)
    assert np.abs(naive - fin[0]).max() > 0.1 * np.abs(fin).max()


def test_chunk_transition_from_the_chunked_quantities():
    """A chunk's transition in the chunked form's terms,
    M_c = Diag(e^{g_C}) - K_bar^T W  (W = (I + A_kk)^-1 diag(beta) (k e^g),
    K_bar = k e^{g_C - g}), equals the product of its tokens' transitions."""
    _, k, _, la, beta, _ = _inputs(64, 2, 16, seed=10)
    M_tok = orc.segment_transition(k, la, beta)
    C = 64
    for h in range(2):
        kh, bh = k[:, h], beta[:, h]
        g = np.cumsum(la[:, h], axis=0)
        decay = np.exp(g[:, None, :] - g[None, :, :])                     # [r, i, c]
        A_kk = np.tril(bh[:, None] * np.einsum("rc,ic,ric->ri", kh, kh, decay), -1)
        W = np.linalg.solve(np.eye(C) + A_kk, bh[:, None] * (kh * np.exp(g)))
        K_bar = kh * np.exp(g[-1][None, :] - g)
        M_c = np.diag(np.exp(g[-1])) - K_bar.T @ W
        assert np.allclose(M_c, M_tok[h], rtol=1e-10, atol=1e-12)
