"""Pins of the counter-causal surprise oracle (oracle/counter_causal.py) to closed forms, an
independent reversed-sequence formulation and exhaustive enumeration (no GPU)."""
import itertools
import math

import numpy as np
import pytest

from oracle import counter_causal as cc


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def test_second_to_last_token_attends_only_to_the_last():
    rng = np.random.default_rng(1)
    K, V, Q = _rand(rng, 2, 9, 16), _rand(rng, 2, 9, 16), _rand(rng, 4, 9, 16)
    o = cc.cc_attention(K, V, Q)
    for h in range(4):
        assert np.allclose(o[7, h], V[h // 2, 8], atol=1e-14)  # one visible token: weight 1
        assert np.all(o[8, h] == 0.0)                          # the last token sees nothing


def test_equal_future_keys_average_the_future_values():
    rng = np.random.default_rng(2)
    n, d = 12, 8
    K = np.tile(_rand(rng, 1, 1, d), (1, n, 1))
    V = _rand(rng, 1, n, d)
    o = cc.cc_attention(K, V, _rand(rng, 1, n, d))
    for i in range(n - 1):
        assert np.allclose(o[i, 0], V[0, i + 1:].mean(0), atol=1e-13)


def test_matches_a_strictly_causal_pass_over_the_reversed_sequence():
    """Position i seeing j > i is, with the token order reversed, a strictly causal mask (each
    position sees the earlier ones only): an independent formulation with a full masked score
    matrix."""
    rng = np.random.default_rng(3)
    n, d = 10, 8
    K, V, Q = _rand(rng, 1, n, d), _rand(rng, 1, n, d), _rand(rng, 1, n, d)
    Kr, Vr, Qr = K[0, ::-1], V[0, ::-1], Q[0, ::-1]
    S = Qr @ Kr.T / math.sqrt(d)
    S = np.where(np.tril(np.ones((n, n)), k=-1) > 0, S, -np.inf)
    o_rev = np.zeros((n, d))
    for i in range(1, n):
        a = np.exp(S[i, :i] - S[i, :i].max())
        o_rev[i] = a @ Vr[:i] / a.sum()
    o = cc.cc_attention(K, V, Q)
    assert np.allclose(o[:, 0], o_rev[::-1], atol=1e-13)


def test_projection_and_unembedding_with_a_permutation_and_one_hot_rows():
    """W_O a (non-symmetric) permutation and W_U one-hot rows: logit_i = h_i[x_i] + o_i[P^-1 x_i],
    so a transposed projection or a wrong row of W_U fails."""
    rng = np.random.default_rng(4)
    n, hq, d = 7, 2, 4
    dm = hq * d
    perm = rng.permutation(dm)
    W_O = np.zeros((dm, dm))
    W_O[np.arange(dm), perm] = 1.0          # (W_O x)[m] = x[perm[m]]
    W_U = np.eye(dm)                        # vocab = d_model, row v = e_v
    X = rng.integers(0, dm, size=n)
    o = _rand(rng, n, hq, d)
    H = _rand(rng, n, dm)
    z = cc.cc_logits(o, H, W_O, W_U, X)
    flat = o.reshape(n, -1)
    assert np.allclose(z, H[np.arange(n), X] + flat[np.arange(n), perm[X]], atol=1e-14)


def test_sinks_and_the_last_token_carry_the_maximum_surprise():
    rng = np.random.default_rng(5)
    n, d, dm = 11, 8, 16
    s = cc.cc_surprise(_rand(rng, 1, n, d), _rand(rng, 1, n, d), _rand(rng, 2, n, d),
                       _rand(rng, n, dm), _rand(rng, dm, 2 * d), _rand(rng, 50, dm),
                       rng.integers(0, 50, size=n), sink=3)
    assert np.all(np.isinf(s[:3])) and np.isinf(s[-1]) and np.all(np.isfinite(s[3:-1]))
    kept = cc.cc_select(s, 6)
    assert {0, 1, 2, n - 1} <= set(kept.tolist())


@pytest.mark.parametrize("seed", range(6))
def test_select_matches_exhaustive_enumeration(seed):
    """The kept set maximises the total surprise; among maximisers with equal scores the lower
    positions win (lexicographically smallest set of positions among the ties)."""
    rng = np.random.default_rng(10 + seed)
    n = int(rng.integers(4, 11))
    J = int(rng.integers(1, n))
    s = rng.integers(0, 4, size=n).astype(np.float64)  # many ties
    best = None
    for sub in itertools.combinations(range(n), J):
        key = (sorted((-s[i] for i in sub)), sub)      # highest values first, then lower positions
        if best is None or key < best[0]:
            best = (key, sub)
    assert cc.cc_select(s, J).tolist() == list(best[1])
    assert cc.cc_select(s, n).tolist() == list(range(n))


def test_row_evaluation_matches_the_whole_sequence():
    """Evaluating selected positions (used at full sizes) gives the same rows as the whole pass."""
    rng = np.random.default_rng(6)
    K, V, Q = _rand(rng, 2, 15, 8), _rand(rng, 2, 15, 8), _rand(rng, 6, 15, 8)
    rows = [14, 0, 7, 13, 3]
    assert np.array_equal(cc.cc_attention_rows(K, V, Q, rows), cc.cc_attention(K, V, Q)[rows])


def _stream(rng, T, hkv=1, hq=2, d=8, dm=12, vocab=40, zero_v=False):
    K, Q = _rand(rng, hkv, T, d), _rand(rng, hq, T, d)
    V = np.zeros((hkv, T, d)) if zero_v else _rand(rng, hkv, T, d)
    return (K, V, Q, _rand(rng, T, dm), _rand(rng, dm, hq * d), _rand(rng, vocab, dm),
            rng.integers(0, vocab, size=T))


@pytest.mark.parametrize("seed,J,h,sink,chunks", [
    (0, 6, 3, 1, [1, 2] * 10 + [3] * 4),      # 42 tokens, refreshes after every 3rd
    (1, 9, 4, 2, [4] * 12),
    (2, 5, 1, 0, [1] * 30),
    (3, 12, 6, 3, [2, 1, 3] * 10),
])
def test_cycle_with_context_free_surprise_keeps_the_global_best(seed, J, h, sink, chunks):
    """V = 0 makes every attention output 0, so each token's surprise is the fixed
    -W_U[x_i].h_i. A token evicted at some refresh was beaten by J - 1 - sink kept tokens, which
    only ever make way for better ones, so the final memory is: the sinks, the final refresh's
    last token, and the J - 1 - sink best of the other tokens (equal: the lower position)."""
    rng = np.random.default_rng(40 + seed)
    T = sum(chunks)
    K, V, Q, H, W_O, W_U, X = _stream(rng, T, zero_v=True)
    mems = cc.cc_cycle(K, V, Q, H, W_O, W_U, X, J, h, sink, chunks)
    assert len(mems) == T // h
    last = T - 1 - (T % h)                              # the last token of the final refresh
    seen = last + 1
    score = -np.einsum("tm,tm->t", W_U[X[:seen]], H[:seen])
    others = [i for i in range(sink, seen) if i != last]
    best = sorted(others, key=lambda i: (-score[i], i))[:J - 1 - sink]
    assert mems[-1].tolist() == sorted(list(range(sink)) + [last] + best)


def test_cycle_invariants_and_no_eviction_below_the_budget():
    rng = np.random.default_rng(50)
    J, h, sink = 7, 3, 2
    chunks = [1, 2, 3, 1, 1, 1, 2, 1, 3, 3, 3]
    K, V, Q, H, W_O, W_U, X = _stream(rng, sum(chunks))
    mems = cc.cc_cycle(K, V, Q, H, W_O, W_U, X, J, h, sink, chunks)
    t = 0
    for k, m in enumerate(mems):
        t = (k + 1) * h
        assert len(m) == min(J, t)
        assert np.all(np.diff(m) > 0)                   # ascending, distinct
        assert set(range(sink)) <= set(m.tolist())      # system-prompt slots never evicted
        assert t - 1 in m                               # the refresh's last token always kept
    # a budget that holds everything evicts nothing
    all_mems = cc.cc_cycle(K, V, Q, H, W_O, W_U, X, 100, h, sink, chunks)
    assert all_mems[-1].tolist() == list(range(len(mems) * h))
