"""Pins of the fp64 oracle against facts fixed by the pages and by mathematics (no GPU).

Each test ties one oracle routine to something other than itself: brute-force deletion of a
token with renormalisation, closed forms, invariants, special cases that reduce to a textbook or
library routine, and exhaustive enumeration on tiny inputs.

LORE-KV project page, Method: "Reliability weights" (Eqs. 2-4, 10), "Projected deletion score"
(Eqs. 5-7), "Evict and decode" (Eq. 8), Hyperparameters table. H2O summary: Section 2.1,
Definitions 2.1/2.2, Section 4.1 (Algorithm 1, linear h), Appendix A.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------------------------------
# Reliability (Eqs. 2-4, 10)
# ------------------------------------------------------------------------------------------
def test_uniform_logits_entropy_is_log_vocab_and_centered_score_is_zero():
    for V in (2, 7, 1024):
        lse, H, logq = oracle.row_stats(np.zeros(V), 3 % V)
        assert abs(H - math.log(V)) < 1e-12
        assert abs(logq + math.log(V)) < 1e-12
        assert abs(logq + H) < 1e-12  # c_u = 0


def test_centered_score_has_zero_conditional_mean():
    rng = np.random.default_rng(1)
    for V in (3, 50, 400):
        z = 2.0 * rng.standard_normal(V)
        stats = [oracle.row_stats(z, y) for y in range(V)]
        H = stats[0][1]
        p = np.array([math.exp(s[2]) for s in stats])
        c = np.array([s[2] + s[1] for s in stats])
        assert abs(p.sum() - 1.0) < 1e-12
        assert abs(float(np.dot(p, c))) < 1e-12          # E_{y~q}[c] = 0 (the page's Eq. 3 claim)
        # independent library routines for the same quantities
        assert abs(stats[0][0] - scipy.special.logsumexp(z)) < 1e-12
        assert abs(H - scipy.stats.entropy(scipy.special.softmax(z))) < 1e-12


def test_row_stats_with_masked_logits_equal_the_restricted_vocabulary():
    """Logits of -inf (masked tokens) have probability 0 and contribute 0 log 0 = 0 to H: the
    row's lse, H and log q(y) equal those of the row with the masked entries removed."""
    rng = np.random.default_rng(4)
    z = 2.0 * rng.standard_normal(300)
    mask = rng.random(300) < 0.3
    y = int(np.flatnonzero(~mask)[7])
    zm = z.copy()
    zm[mask] = -np.inf
    got = oracle.row_stats(zm, y)
    keep = np.flatnonzero(~mask)
    want = oracle.row_stats(z[keep], int(np.searchsorted(keep, y)))
    assert np.all(np.isfinite(got))
    assert np.allclose(got, want, rtol=1e-13, atol=1e-13)
    assert abs(got[0] - scipy.special.logsumexp(z[keep])) < 1e-12


def test_row_stats_invariant_to_logit_shift():
    rng = np.random.default_rng(2)
    z = rng.standard_normal(300)
    a = oracle.row_stats(z, 17)
    b = oracle.row_stats(z + 123.25, 17)
    assert abs(a[1] - b[1]) < 1e-12 and abs(a[2] - b[2]) < 1e-12
    assert abs((b[0] - a[0]) - 123.25) < 1e-10


def _rand_rel(rng, M, T, V, LH=3, d=8):
    logits = 2.0 * rng.standard_normal((M * T, V))
    y = rng.integers(0, V, size=M * T).astype(np.int32)
    ql = rng.standard_normal((LH, M * T, d))
    return logits, y, ql


def test_omega_is_a_distribution_and_single_trajectory_gets_weight_one():
    rng = np.random.default_rng(3)
    logits, y, ql = _rand_rel(rng, 4, 8, 64)
    r = oracle.reliability(logits, y, ql, 4, 8, 1.0, 1.3, 0.0)
    assert abs(r["omega"].sum() - 1.0) < 1e-12 and np.all(r["omega"] > 0)
    r1 = oracle.reliability(logits[:8], y[:8], ql[:, :8], 1, 8, 1.0, 1.0, 0.3)
    assert r1["omega"].tolist() == [1.0]


def test_omega_without_disagreement_ignores_lookahead_queries():
    rng = np.random.default_rng(4)
    logits, y, ql = _rand_rel(rng, 4, 8, 64)
    a = oracle.reliability(logits, y, ql, 4, 8, 1.0, 1.3, 0.0)["omega"]
    b = oracle.reliability(logits, y, rng.standard_normal(ql.shape), 4, 8, 1.0, 1.3, 0.0)["omega"]
    assert np.array_equal(a, b)


def test_omega_permutes_with_trajectories():
    rng = np.random.default_rng(5)
    M, T = 4, 3
    logits, y, ql = _rand_rel(rng, M, T, 40)
    perm = [2, 0, 3, 1]
    rows = np.concatenate([np.arange(m * T, m * T + T) for m in perm])
    a = oracle.reliability(logits, y, ql, M, T, 1.0, 1.0, 0.3)["omega"]
    b = oracle.reliability(logits[rows], y[rows], ql[:, rows], M, T, 1.0, 1.0, 0.3)["omega"]
    assert np.allclose(a[perm], b, rtol=1e-12, atol=0)


def test_omega_equal_trajectories_are_uniform():
    rng = np.random.default_rng(6)
    M, T, V = 4, 2, 30
    logits1 = rng.standard_normal((T, V))
    y1 = rng.integers(0, V, size=T).astype(np.int32)
    logits = np.tile(logits1, (M, 1))
    y = np.tile(y1, M)
    ql = np.tile(rng.standard_normal((2, T, 8)), (1, M, 1))
    om = oracle.reliability(logits, y, ql, M, T, 1.0, 1.0, 0.3)["omega"]
    assert np.allclose(om, 0.25, rtol=0, atol=1e-15)


def test_disagreement_geometry_golden():
    """Three trajectories whose mean queries are e1, e1, e2 (cosines 1, 0, 0): D = (0.5, 0.5, 1),
    standardised -> (-1/sqrt2, -1/sqrt2, sqrt2). Fixture: tests/golden/disagreement_geometry.json."""
    with open(os.path.join(GOLDEN, "disagreement_geometry.json")) as f:
        gold = json.load(f)
    M, T, d = 3, 2, 4
    ql = np.zeros((1, M * T, d))
    ql[0, 0:2, 0] = [0.5, 1.5]   # mean e1
    ql[0, 2:4, 0] = [2.0, 0.0]   # mean e1
    ql[0, 4:6, 1] = [3.0, 1.0]   # mean 2 e2
    logits = np.zeros((M * T, 5))
    y = np.zeros(M * T, dtype=np.int32)
    r = oracle.reliability(logits, y, ql, M, T, 0.0, 0.0, 1.0)
    assert np.allclose(r["Dhat"], gold["Dhat"], rtol=0, atol=1e-12)
    # R = -Dhat when beta = gamma = 0, lambda_D = 1
    assert np.allclose(r["R"], -np.array(gold["Dhat"]), rtol=0, atol=1e-12)


# ------------------------------------------------------------------------------------------
# Gram / Cholesky (e = ||W_O Delta o|| evaluated as ||L^T Delta o||)
# ------------------------------------------------------------------------------------------
def test_cholesky_reconstructs_gram_and_reproduces_projection_norm():
    rng = np.random.default_rng(7)
    d_model, Hq, d = 48, 3, 8
    W = rng.standard_normal((d_model, Hq * d)) / math.sqrt(d_model)
    for h in range(Hq):
        G, L, st = oracle.gram_cholesky(W, d, h)
        assert st == oracle.OK
        assert np.allclose(np.tril(L), L, atol=0)
        assert np.linalg.norm(L @ L.T - G) <= 1e-12 * np.linalg.norm(G)
        Wh = W[:, h * d:(h + 1) * d]
        for _ in range(5):
            x = rng.standard_normal(d)
            direct = np.linalg.norm(Wh @ x)
            assert abs(np.linalg.norm(L.T @ x) - direct) <= 1e-12 * direct


def test_orthonormal_projection_gives_identity_factor_and_head_columns_are_used():
    rng = np.random.default_rng(8)
    d_model, d = 32, 8
    blocks = []
    for h in range(3):
        Qm, _ = np.linalg.qr(rng.standard_normal((d_model, d)))
        blocks.append((h + 1.0) * Qm)      # head h: columns scaled by (h+1)
    W = np.concatenate(blocks, axis=1)
    for h in range(3):
        G, L, st = oracle.gram_cholesky(W, d, h)
        assert st == oracle.OK
        assert np.allclose(L, (h + 1.0) * np.eye(d), atol=1e-12)


def test_rank_deficient_projection_is_not_positive_definite():
    rng = np.random.default_rng(9)
    W = rng.standard_normal((4, 8))           # d_model < d: G has rank 4
    _, _, st = oracle.gram_cholesky(W, 8, 0)
    assert st == oracle.ENOTPD


# ------------------------------------------------------------------------------------------
# Projected deletion score (Eqs. 5-7) against brute-force deletion
# ------------------------------------------------------------------------------------------
def _tiny_unit(rng, n=24, d=8, g=2, w=4, M=2, T=2, d_model=16):
    K = rng.standard_normal((n, d))
    V = rng.standard_normal((n, d))
    QW = rng.standard_normal((g, w, d)) * 1.5
    QL = rng.standard_normal((g, M * T, d)) * 1.5
    W = rng.standard_normal((d_model, g * d)) / math.sqrt(d_model)
    Lf = np.stack([oracle.gram_cholesky(W, d, h)[1] for h in range(g)])
    return K, V, QW, QL, W, Lf


def _visible(n, w, qidx, causal):
    """Tokens query qidx may attend: window query r sits at position n-w+r (causal reading)."""
    if qidx < w and causal:
        return np.arange(n - w + qidx + 1)
    return np.arange(n)


def _brute_force_e(K, V, QW, QL, W, causal, M, T):
    """e_{q,i} by deleting token i, renormalising and recomputing the attention output,
    then projecting the change through the d_model-wide W_O^h."""
    n, d = K.shape
    g, w = QW.shape[:2]
    nq = w + M * T
    E = np.zeros((g, nq, n))
    A = np.zeros((g, nq, n))
    for h in range(g):
        Wh = W[:, h * d:(h + 1) * d]
        for qi in range(nq):
            q = QW[h, qi] if qi < w else QL[h, qi - w]
            vis = _visible(n, w, qi, causal)
            s = K[vis] @ q / math.sqrt(d)
            a = np.exp(s - s.max())
            a /= a.sum()
            o = a @ V[vis]
            A[h, qi, vis] = a
            for j, i in enumerate(vis):
                rest = np.delete(np.arange(len(vis)), j)
                s2 = s[rest]
                a2 = np.exp(s2 - s2.max())
                a2 /= a2.sum()
                o2 = a2 @ V[vis[rest]]
                E[h, qi, i] = np.linalg.norm(Wh @ (o - o2))
    return E, A


@pytest.mark.parametrize("causal", [1, 0])
def test_projected_deletion_matches_brute_force_deletion(causal):
    rng = np.random.default_rng(10 + causal)
    M, T = 2, 2
    K, V, QW, QL, W, Lf = _tiny_unit(rng, M=M, T=T)
    E_bf, A = _brute_force_e(K, V, QW, QL, W, causal, M, T)
    r = oracle.lorekv_unit(K, V, QW, QL, Lf, [0.5, 0.5], M=M, T=T, sink=2, lambda_L=1.0,
                           eps=0.0, window_causal=causal, want=("E", "lse", "o"))
    assert np.allclose(r["E"], E_bf, rtol=1e-12, atol=1e-14)
    # eps = 1e-6: e scales by (1-a)/(1-a+eps) relative to the exact deletion
    r2 = oracle.lorekv_unit(K, V, QW, QL, Lf, [0.5, 0.5], M=M, T=T, sink=2, lambda_L=1.0,
                            eps=1e-6, window_causal=causal, want=("E",))
    corr = np.where(A > 0, (1 - A) / (1 - A + 1e-6), 0.0)
    assert np.allclose(r2["E"], E_bf * corr, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("target", [0.999, 1 - 1e-7])
def test_projected_deletion_matches_brute_force_when_one_token_dominates(target):
    """The peaked regime: one non-protected token takes a of about 0.999 (and 1 - 1e-7) of a
    query's attention. The oracle's difference form still reproduces brute-force deletion there,
    where 1 - a and v_i - o_q are small differences of large numbers."""
    rng = np.random.default_rng(17)
    M, T = 2, 2
    K, V, QW, QL, W, Lf = _tiny_unit(rng, M=M, T=T)
    n, d = K.shape
    h, qi, p = 1, 5, 9                       # lookahead query 1 of head 1, token 9
    q = QL[h, qi - QW.shape[1]]
    s = K @ q / math.sqrt(d)
    rest = np.delete(np.arange(n), p)
    R = np.exp(s[rest] - s[rest].max()).sum() * math.exp(s[rest].max())
    # k_p <- k_p + beta q/|q| so that a_{q,p} = target
    want = math.log(target / (1 - target) * R)
    K[p] += (want - s[p]) * math.sqrt(d) / (q @ q) * q
    E_bf, A = _brute_force_e(K, V, QW, QL, W, 0, M, T)
    assert abs(A[h, qi, p] - target) < 1e-9
    r = oracle.lorekv_unit(K, V, QW, QL, Lf, [0.5, 0.5], M=M, T=T, sink=2, lambda_L=1.0,
                           eps=0.0, window_causal=0, want=("E",))
    # both sides subtract nearly equal fp64 vectors: brute force o - o_without_i loses digits as
    # 1/a for tiny a, the difference form v_i - o_q as 1/(1 - a) near a = 1
    rtol = 1e-10 + 1e-14 / np.maximum(np.minimum(A, 1 - A), 1e-300)
    assert np.all(np.abs(r["E"] - E_bf) <= rtol * np.abs(E_bf) + 1e-15)
    assert abs(r["E"][h, qi, p] / E_bf[h, qi, p] - 1) < 1e-14 / (1 - target)


def test_aggregation_weights_window_and_trajectories():
    """S_i = mean over window queries + lambda_L sum_m omega_m mean over trajectory m's queries,
    means taken over all g query heads; protected tokens report 0."""
    rng = np.random.default_rng(12)
    M, T, w, sink = 3, 2, 4, 2
    K, V, QW, QL, W, Lf = _tiny_unit(rng, n=28, w=w, M=M, T=T)
    E_bf, _ = _brute_force_e(K, V, QW, QL, W, 1, M, T)
    n, g = K.shape[0], QW.shape[0]
    omega = np.array([0.2, 0.5, 0.3])
    for lam in (0.0, 1.0, 0.7):
        S = oracle.lorekv_unit(K, V, QW, QL, Lf, omega, M=M, T=T, sink=sink, lambda_L=lam,
                               eps=0.0)
        win = E_bf[:, :w, :].mean(axis=(0, 1))
        look = sum(omega[m] * E_bf[:, w + m * T:w + (m + 1) * T, :].mean(axis=(0, 1))
                   for m in range(M))
        want = win + lam * look
        want[:sink] = 0
        want[n - w:] = 0
        assert np.allclose(S, want, rtol=1e-12, atol=1e-15)


def test_scores_invariant_to_trajectory_order():
    rng = np.random.default_rng(13)
    M, T = 4, 2
    K, V, QW, QL, W, Lf = _tiny_unit(rng, M=M, T=T)
    omega = np.array([0.1, 0.2, 0.3, 0.4])
    perm = [3, 1, 0, 2]
    rows = np.concatenate([np.arange(m * T, m * T + T) for m in perm])
    a = oracle.lorekv_unit(K, V, QW, QL, Lf, omega, M=M, T=T, sink=2, lambda_L=1.0, eps=1e-6)
    b = oracle.lorekv_unit(K, V, QW, QL[:, rows], Lf, omega[perm], M=M, T=T, sink=2,
                           lambda_L=1.0, eps=1e-6)
    assert np.allclose(a, b, rtol=1e-12, atol=0)


def test_equal_keys_give_uniform_attention_and_identity_factor_gives_plain_norm():
    rng = np.random.default_rng(14)
    n, d, g, w, M, T = 20, 6, 1, 4, 2, 2
    K = np.tile(rng.standard_normal(d), (n, 1))
    V = rng.standard_normal((n, d))
    QW = rng.standard_normal((g, w, d))
    QL = rng.standard_normal((g, M * T, d))
    Lf = np.eye(d)[None]
    eps = 1e-6
    r = oracle.lorekv_unit(K, V, QW, QL, Lf, [0.5, 0.5], M=M, T=T, sink=1, lambda_L=1.0,
                           eps=eps, window_causal=0, want=("E", "lse", "o"))
    vbar = V.mean(axis=0)
    for q in range(w + M * T):
        qv = QW[0, q] if q < w else QL[0, q - w]
        assert abs(r["lse"][0, q] - (math.log(n) + K[0] @ qv / math.sqrt(d))) < 1e-12
        assert np.allclose(r["o"][0, q], vbar, rtol=0, atol=1e-13)
        a = 1.0 / n
        want = a / (1 - a + eps) * np.linalg.norm(V - vbar, axis=1)
        assert np.allclose(r["E"][0, q], want, rtol=1e-12, atol=0)


def test_causal_window_queries_do_not_see_later_tokens():
    rng = np.random.default_rng(15)
    K, V, QW, QL, W, Lf = _tiny_unit(rng)
    n, w = K.shape[0], QW.shape[1]
    r = oracle.lorekv_unit(K, V, QW, QL, Lf, [0.5, 0.5], M=2, T=2, sink=2, lambda_L=1.0,
                           eps=1e-6, want=("E",))
    for qi in range(w):
        assert np.all(r["E"][:, qi, n - w + qi + 1:] == 0)
        assert np.all(r["E"][:, qi, :n - w + qi + 1] > 0)


# ------------------------------------------------------------------------------------------
# Chunked top-B selection (Eq. 8) against exhaustive enumeration
# ------------------------------------------------------------------------------------------
def test_select_matches_exhaustive_enumeration():
    rng = np.random.default_rng(16)
    sink, w, chunk = 2, 3, 4
    for trial in range(40):
        nch = int(rng.integers(1, 13))
        n = sink + w + chunk * nch
        S = rng.integers(0, 4, size=n).astype(np.float64)  # small integers -> many ties
        cs = np.array([S[sink + c * chunk: sink + (c + 1) * chunk].mean() for c in range(nch)])
        for k in range(0, nch + 2):
            kept = oracle.select(S, sink=sink, w=w, chunk=chunk, B=k * chunk)
            if k >= nch:
                assert kept.tolist() == list(range(n))
                continue
            best = None
            for comb in itertools.combinations(range(nch), k):   # lexicographic order
                tot = cs[list(comb)].sum()
                if best is None or tot > best[0] + 1e-12:
                    best = (tot, comb)
            want = list(range(sink))
            for c in best[1]:
                want += list(range(sink + c * chunk, sink + (c + 1) * chunk))
            want += list(range(n - w, n))
            assert kept.tolist() == want, (trial, k)


def test_select_rejects_ragged_shapes():
    with pytest.raises(ValueError):
        oracle.select(np.zeros(31), sink=4, w=4, chunk=4, B=8)     # 23 not divisible by 4
    with pytest.raises(ValueError):
        oracle.select(np.zeros(32), sink=4, w=4, chunk=4, B=6)     # B not a multiple of 4


# ------------------------------------------------------------------------------------------
# H2O (Section 2.1, Definitions 2.1/2.2, Section 4.1, Appendix A)
# ------------------------------------------------------------------------------------------
def test_prefill_accumulated_scores_equal_keys_are_harmonic_tails():
    """All keys equal: query i spreads 1/(i+1) over tokens 0..i, so acc_j = sum_{i=j}^{P-1} 1/(i+1)."""
    rng = np.random.default_rng(17)
    P, d = 40, 8
    K = np.tile(rng.standard_normal(d), (P, 1))
    Q = rng.standard_normal((P, d))
    acc = oracle.h2o_prefill_acc(K, Q)
    want = np.array([sum(1.0 / (i + 1) for i in range(j, P)) for j in range(P)])
    assert np.allclose(acc, want, rtol=1e-13, atol=0)
    acc2 = oracle.h2o_prefill_acc(rng.standard_normal((P, d)), Q)
    assert abs(acc2.sum() - P) < 1e-12


def test_zero_key_identity_of_constrained_attention():
    """Definition 2.2: zeroing the keys of evicted tokens and subtracting their spurious exp(0)=1
    terms from the normaliser gives the softmax over the retained tokens."""
    rng = np.random.default_rng(18)
    i, d = 30, 8
    K = rng.standard_normal((i, d))
    V = rng.standard_normal((i, d))
    q = rng.standard_normal(d)
    keep = np.sort(rng.choice(i, size=12, replace=False))
    Kz = np.zeros_like(K)
    Kz[keep] = K[keep]
    ex = np.exp(Kz @ q / math.sqrt(d))
    mask = np.ones(i)
    mask[keep] = 0
    D = (ex - mask).sum()
    o_constrained = (ex * (1 - mask)) / D
    p, out = oracle.h2o_attend(K[keep], V[keep], q)
    assert np.allclose(o_constrained[keep], p, rtol=1e-12, atol=0)
    assert np.allclose(out, o_constrained @ V, rtol=1e-12, atol=1e-15)


def test_greedy_eviction_is_argmin_of_accumulated_score():
    """With linear h, argmax_v F(G \\ {v}) = argmin_v acc_v over the candidates; recent tokens
    (the k_t/2 most recent) are never candidates; ties go to the oldest."""
    rng = np.random.default_rng(19)
    for trial in range(200):
        t = int(rng.integers(20, 80))
        k, r = oracle.h2o_budget(t, 0.2)
        cnt = k + 1
        pos = np.sort(rng.choice(np.arange(t - 1), size=cnt - 1, replace=False)).tolist() + [t - 1]
        pos = np.array(pos, dtype=np.int32)
        acc = rng.integers(0, 5, size=cnt).astype(np.float64) / 4.0
        ev = oracle.h2o_evict(pos, acc, t, 0.2)
        assert ev.sum() == 1
        cands = [j for j in range(cnt) if pos[j] < t - r]
        F = lambda keep: sum(acc[j] for j in keep)           # linear h
        best = max(cands, key=lambda v: (F([j for j in range(cnt) if j != v]), -pos[v]))
        assert np.flatnonzero(ev).tolist() == [best]


@pytest.mark.parametrize("hname", ["sqrt", "log"])
def test_greedy_eviction_with_concave_score_function(hname):
    """F_score(T) = h(sum_{s in T} acc_s) with a non-decreasing concave h (H2O summary, "Define
    the score function": sqrt(z + 1), log(z + 1)): argmax_v h(total - acc_v) over the candidates is
    the same token as with linear h, because h is increasing; the eviction the kernels implement
    (argmin acc, oldest on ties) therefore serves every such h."""
    h = {"sqrt": lambda z: np.sqrt(z + 1.0), "log": lambda z: np.log(z + 1.0)}[hname]
    rng = np.random.default_rng(23)
    for trial in range(200):
        t = int(rng.integers(20, 80))
        k, r = oracle.h2o_budget(t, 0.2)
        cnt = k + 1
        pos = np.sort(rng.choice(np.arange(t - 1), size=cnt - 1, replace=False)).tolist() + [t - 1]
        pos = np.array(pos, dtype=np.int32)
        acc = rng.integers(0, 5, size=cnt).astype(np.float64) / 4.0
        ev = oracle.h2o_evict(pos, acc, t, 0.2)
        cands = [j for j in range(cnt) if pos[j] < t - r]
        F = lambda keep: h(sum(acc[j] for j in keep))
        best = max(cands, key=lambda v: (F([j for j in range(cnt) if j != v]), -pos[v]))
        assert np.flatnonzero(ev).tolist() == [best]


def test_h2o_decode_invariants():
    rng = np.random.default_rng(20)
    P, d, steps, frac = 64, 16, 64, 0.2
    K = rng.standard_normal((P, d))
    V = rng.standard_normal((P, d))
    Q = rng.standard_normal((P, d))
    u = oracle.H2OUnit(K, V, Q, frac, P + steps)
    k0, r0 = oracle.h2o_budget(P, frac)
    assert len(u.pos) == k0 and set(range(P - r0, P)) <= set(u.pos.tolist())
    for s in range(steps):
        before = set(u.pos.tolist())
        out, evicted, pre = u.step(rng.standard_normal(d), rng.standard_normal(d),
                                   rng.standard_normal(d))
        t = P + s + 1
        k, r = oracle.h2o_budget(t, frac)
        assert len(u.pos) == k                                 # |S_i| = k_t
        assert len(evicted) <= 1                               # at most one eviction per step
        assert set(range(t - r, t)) <= set(u.pos.tolist())     # recent window kept
        assert len(set(u.pos.tolist()) - before) <= 1          # |S_i \ S_{i-1}| <= 1
        assert abs(u.full_acc.sum() - u.queries) < 1e-12       # softmax rows sum to one
