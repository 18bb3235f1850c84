"""Pins of the fp64 block-verifier and draft-sampler oracles.

The rule ("Unlocking Lossless Speedups in LLMs via Discrete Diffusion",
aifromscratch.in, section "The Psi-Spec Sampler"; "Uno Uses Discrete
Diffusion to Accelerate LLMs Without Loss", cctest.ai, section "What
'lossless' means here"): drafts are accepted while u_i < min(1, p_i/q_i);
at the first rejection one token is drawn from max(0, p - q) normalised; the
emitted tokens are distributed exactly as the AR model's.

Pins, none of which re-types the oracle's procedure:
  * hand-worked golden examples (tests/golden/verify_tiny.txt, race_tiny.txt);
  * q == p accepts every draft; disjoint supports accept none;
  * the acceptance threshold sits at min(1, p/q) (strict '<');
  * closed form E[n] = sum_{k=1}^{K} prod_{i<k} alpha_i, alpha_i = sum_v min(p_i, q_i);
  * losslessness: chi-square of every emitted position against p_i, with
    drafts drawn by numpy from q (independent of the oracle);
  * the resampled token follows max(0, p - q)/S; the draft sampler follows q;
  * status codes for bad drafts and non-finite logits.
"""
import numpy as np
import pytest
from scipy import stats

from conftest import read_golden

TWO24 = float(1 << 24)


def _u_accept(rng, shape):
    return (rng.integers(0, 1 << 24, size=shape) / TWO24).astype(np.float32)


def _u_race(rng, shape):
    return (rng.integers(1, 1 << 24, size=shape) / TWO24).astype(np.float32)


def _softmax(l):
    l = np.asarray(l, np.float64)
    e = np.exp(l - l.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def test_golden_verify_tiny(oracle_mod):
    g = read_golden("verify_tiny.txt")
    V, K = int(g["V"][0]), int(g["K"][0])
    p = np.log(np.array([g["p0"], g["p1"]], np.float64)).astype(np.float32)[None]
    q = np.log(np.array([g["q0"], g["q1"]], np.float64)).astype(np.float32)[None]
    d = np.array(g["draft"], np.int32)[None]
    ua = np.array(g["u_accept"], np.float32)[None]
    ur = np.array(g["u_resample"], np.float32)[None]
    r = oracle_mod.verify_block(p, q, d, ua, ur)
    assert r.n_accepted[0] == g["n_accepted"][0]
    assert r.n_emitted[0] == g["n_emitted"][0]
    assert r.out_tokens[0].tolist() == [int(t) for t in g["out_tokens"]]
    assert r.status[0] == 0 and V == 3 and K == 2


def test_golden_race_tiny(oracle_mod):
    g = read_golden("race_tiny.txt")
    logits = np.log(np.array(g["q"]))[None].astype(np.float32)
    u = np.array(g["u"], np.float32)[None]
    tok, st, _ = oracle_mod.draft_sample(logits, u)
    assert tok[0] == int(g["token"][0]) and st[0] == 0


@pytest.mark.parametrize("bonus", [False, True])
def test_q_equals_p_accepts_everything(oracle_mod, bonus):
    rng = np.random.default_rng(5)
    Bn, K, V = 64, 5, 50
    Kp = K + 1 if bonus else K
    p = (rng.standard_normal((Bn, Kp, V)) * 3).astype(np.float32)
    q = p[:, :K].copy()
    d = rng.integers(0, V, size=(Bn, K)).astype(np.int32)
    r = oracle_mod.verify_block(p, q, d, _u_accept(rng, (Bn, K)), _u_race(rng, (Bn, V)))
    assert (r.n_accepted == K).all()
    assert (r.n_emitted == Kp).all()
    np.testing.assert_array_equal(r.out_tokens[:, :K], d)
    if bonus:
        assert ((r.out_tokens[:, K] >= 0) & (r.out_tokens[:, K] < V)).all()
    else:
        assert (r.out_tokens[:, K] == -1).all()


def test_disjoint_supports_accept_nothing(oracle_mod):
    rng = np.random.default_rng(6)
    Bn, K, V = 200, 3, 8
    ninf = -np.inf
    p_row = np.array([0, 1, 2, 0.5, ninf, ninf, ninf, ninf], np.float32)
    q_row = np.array([ninf, ninf, ninf, ninf, 0, 1, 0, -1], np.float32)
    p = np.broadcast_to(p_row, (Bn, K, V)).copy()
    q = np.broadcast_to(q_row, (Bn, K, V)).copy()
    d = rng.integers(4, 8, size=(Bn, K)).astype(np.int32)
    ua = _u_accept(rng, (Bn, K))
    ua[:, 0] = 0.0  # p(x)=0 gives rho=0 and u=0 is not < 0: still rejected
    r = oracle_mod.verify_block(p, q, d, ua, _u_race(rng, (Bn, V)))
    assert (r.n_accepted == 0).all() and (r.n_emitted == 1).all()
    assert ((r.out_tokens[:, 0] >= 0) & (r.out_tokens[:, 0] < 4)).all()
    assert (r.out_tokens[:, 1:] == -1).all()


def test_threshold_at_min_one_ratio(oracle_mod):
    V = 4
    p = np.log(np.array([[[0.4, 0.3, 0.2, 0.1]]])).astype(np.float32)
    q = np.log(np.array([[[0.1, 0.6, 0.2, 0.1]]])).astype(np.float32)
    ur = np.full((1, V), 0.5, np.float32)
    # draft 1: rho = 0.3/0.6 = 0.5
    for u, acc in [(0.4999, 1), (0.5001, 0), (0.0, 1), (0.9, 0)]:
        r = oracle_mod.verify_block(p, q, np.array([[1]], np.int32),
                                    np.array([[u]], np.float32), ur)
        assert r.n_accepted[0] == acc, (u, acc)
        assert abs(r.accept_margin[0, 0] - abs(0.5 - u)) < 1e-6
    # draft 0: rho = 4 >= 1, accepted for the largest u below 1
    r = oracle_mod.verify_block(p, q, np.array([[0]], np.int32),
                                np.array([[1 - 2 ** -24]], np.float32), ur)
    assert r.n_accepted[0] == 1


def _stat_problem(seed, Bn, K, V, Kp, sigma=1.0):
    """Shared distributions per position (distinct across positions), drafts
    drawn by numpy from q, independent uniforms per sequence."""
    rng = np.random.default_rng(seed)
    lp = (rng.standard_normal((Kp, V)) * 1.5).astype(np.float32)
    lq = (lp[:K] + rng.standard_normal((K, V)) * sigma).astype(np.float32)
    P, Q = _softmax(lp), _softmax(lq)
    d = np.stack([rng.choice(V, size=Bn, p=Q[i]) for i in range(K)], axis=1).astype(np.int32)
    p = np.broadcast_to(lp, (Bn, Kp, V)).copy()
    q = np.broadcast_to(lq, (Bn, K, V)).copy()
    return p, q, d, _u_accept(rng, (Bn, K)), _u_race(rng, (Bn, V)), P, Q


@pytest.fixture(scope="module")
def stat_run(oracle_mod):
    Bn, K, V, Kp = 200_000, 3, 8, 4
    p, q, d, ua, ur, P, Q = _stat_problem(123, Bn, K, V, Kp)
    r = oracle_mod.verify_block(p, q, d, ua, ur)
    return dict(r=r, P=P, Q=Q, K=K, V=V, Kp=Kp, Bn=Bn)


def test_closed_form_mean_accepted(stat_run):
    r, P, Q, K = stat_run["r"], stat_run["P"], stat_run["Q"], stat_run["K"]
    alpha = np.minimum(P[:K], Q).sum(axis=1)
    expect = sum(np.prod(alpha[:k]) for k in range(1, K + 1))
    n = r.n_accepted.astype(np.float64)
    z = (n.mean() - expect) / (n.std() / np.sqrt(n.size))
    assert abs(z) < 4.0, (n.mean(), expect, z)
    # and P(n >= k) = prod_{i<k} alpha_i for each k
    for k in range(1, K + 1):
        frac = (r.n_accepted >= k).mean()
        want = np.prod(alpha[:k])
        se = np.sqrt(want * (1 - want) / n.size)
        assert abs(frac - want) < 5 * se + 1e-12, (k, frac, want)


def test_emitted_tokens_follow_p(stat_run):
    """Losslessness: token i, given that it was emitted, is distributed as p_i."""
    r, P, V, Kp = stat_run["r"], stat_run["P"], stat_run["V"], stat_run["Kp"]
    for i in range(Kp):
        sel = r.n_emitted > i
        toks = r.out_tokens[sel, i]
        obs = np.bincount(toks, minlength=V)
        res = stats.chisquare(obs, P[i] * sel.sum())
        assert res.pvalue > 1e-3, (i, res)


def test_resample_follows_residual(stat_run):
    r, P, Q, V, K = stat_run["r"], stat_run["P"], stat_run["Q"], stat_run["V"], stat_run["K"]
    for i in range(K):
        sel = (r.n_accepted == i)
        toks = r.out_tokens[sel, i]
        res_p = np.maximum(P[i] - Q[i], 0.0)
        res_p /= res_p.sum()
        obs = np.bincount(toks, minlength=V)
        support = res_p > 0
        assert obs[~support].sum() == 0
        res = stats.chisquare(obs[support], res_p[support] * sel.sum())
        assert res.pvalue > 1e-3, (i, res)


def test_draft_sampler_follows_softmax(oracle_mod):
    rng = np.random.default_rng(9)
    R, V = 300_000, 8
    lg = (rng.standard_normal(V) * 2).astype(np.float32)
    logits = np.broadcast_to(lg, (R, V)).copy()
    tok, st, _ = oracle_mod.draft_sample(logits, _u_race(rng, (R, V)))
    assert (st == 0).all()
    res = stats.chisquare(np.bincount(tok, minlength=V), _softmax(lg) * R)
    assert res.pvalue > 1e-3, res


def test_no_drafts_is_plain_ar_sampling(oracle_mod):
    """K = 0, Kp = 1: the verifier draws one token from p_0."""
    rng = np.random.default_rng(10)
    Bn, V = 200_000, 8
    lp = (rng.standard_normal(V) * 2).astype(np.float32)
    p = np.broadcast_to(lp, (Bn, 1, V)).copy()
    q = np.zeros((Bn, 0, V), np.float32)
    r = oracle_mod.verify_block(p, q, np.zeros((Bn, 0), np.int32),
                                np.zeros((Bn, 0), np.float32), _u_race(rng, (Bn, V)))
    assert (r.n_accepted == 0).all() and (r.n_emitted == 1).all()
    res = stats.chisquare(np.bincount(r.out_tokens[:, 0], minlength=V), _softmax(lp) * Bn)
    assert res.pvalue > 1e-3, res


def test_status_codes(oracle_mod):
    rng = np.random.default_rng(12)
    Bn, K, V = 5, 2, 16
    p = rng.standard_normal((Bn, K, V)).astype(np.float32)
    q = p.copy()
    d = rng.integers(0, V, size=(Bn, K)).astype(np.int32)
    d[1, 1] = V          # out of range
    d[2, 0] = -1         # out of range
    p[3, 1, 5] = np.nan  # NaN logit
    q[4, 0, :] = -np.inf  # a row with no support
    p[0, 0, 3] = -np.inf  # a single -inf entry is a valid zero probability
    r = oracle_mod.verify_block(p, q, d, _u_accept(rng, (Bn, K)), _u_race(rng, (Bn, V)))
    assert r.status.tolist() == [0, 1, 1, 2, 2]
    assert (r.n_accepted[1:] == 0).all() and (r.n_emitted[1:] == 0).all()
    assert (r.out_tokens[1:] == -1).all()
    assert r.n_accepted[0] == K


def test_empty_batch(oracle_mod):
    r = oracle_mod.verify_block(np.zeros((0, 2, 4), np.float32), np.zeros((0, 2, 4), np.float32),
                                np.zeros((0, 2), np.int32), np.zeros((0, 2), np.float32),
                                np.zeros((0, 4), np.float32))
    assert r.n_accepted.shape == (0,)
