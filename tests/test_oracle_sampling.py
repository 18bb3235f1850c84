"""Pins of the verifier oracle's sampling variants: temperature T and the
single-uniform inverse-CDF resample ("Unlocking Lossless Speedups in LLMs via
Discrete Diffusion", aifromscratch.in, section "The Psi-Spec Sampler": the
speculative-decoding acceptance rule, here with every distribution taken at
temperature T, p = softmax(l_p / T), q = softmax(l_q / T)).

Pins, none of which re-types the oracle's procedure:
  * a hand-worked golden example of the inverse CDF (tests/golden/inverse_cdf_tiny.txt);
  * T = 1 with the race is the plain verifier, output for output;
  * T = 2 equals the plain verifier on halved logits (halving is exact in fp32);
  * losslessness at T != 1: chi-square of every emitted position against
    softmax(l_p / T), drafts drawn by numpy from softmax(l_q / T);
  * the inverse-CDF resample follows max(0, p - q)/S and the emitted tokens follow p;
  * invalid temperatures are rejected.
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


def test_golden_inverse_cdf_tiny(oracle_mod):
    g = read_golden("inverse_cdf_tiny.txt")
    V = int(g["V"][0])
    p = np.log(np.array(g["p"], np.float64)).astype(np.float32)[None, None]
    q = np.log(np.array(g["q"], np.float64)).astype(np.float32)[None, None]
    for u, tok in zip(g["u_resample"], g["tokens"]):
        r = oracle_mod.verify_block_ex(p, q, np.array([[int(g["draft"][0])]], np.int32),
                                       np.array([[g["u_accept"][0]]], np.float32),
                                       np.array([u], np.float32), resample="inverse_cdf")
        assert r.n_accepted[0] == 0 and r.n_emitted[0] == 1
        assert r.out_tokens[0].tolist() == [int(tok), -1], (u, tok)
    pb = np.log(np.array(g["bonus_p"], np.float64)).astype(np.float32)[None, None]
    for u, tok in zip(g["bonus_u"], g["bonus_tokens"]):
        r = oracle_mod.verify_block_ex(pb, np.zeros((1, 0, V), np.float32), np.zeros((1, 0), np.int32),
                                       np.zeros((1, 0), np.float32), np.array([u], np.float32),
                                       resample="inverse_cdf")
        assert r.n_emitted[0] == 1 and r.out_tokens[0, 0] == int(tok), (u, tok)
        assert 0 < r.race_margin[0] < 1


def _problem(seed, Bn, K, V, Kp, T=1.0, sigma=1.0):
    rng = np.random.default_rng(seed)
    lp = (rng.standard_normal((Bn, Kp, V)) * 2).astype(np.float32)
    lq = (lp[:, :K] + rng.standard_normal((Bn, K, V)) * sigma).astype(np.float32)
    Q = _softmax(lq / T)
    d = np.array([[rng.choice(V, p=Q[b, i]) for i in range(K)] for b in range(Bn)], np.int32)
    return lp, lq, d, _u_accept(rng, (Bn, K)), _u_race(rng, (Bn, V))


@pytest.mark.parametrize("Kp", [6, 7])
def test_unit_temperature_race_is_the_plain_verifier(oracle_mod, Kp):
    p, q, d, ua, ur = _problem(31, 64, 6, 300, Kp)
    a = oracle_mod.verify_block(p, q, d, ua, ur)
    b = oracle_mod.verify_block_ex(p, q, d, ua, ur, temperature=1.0, resample="race")
    for f in ("n_accepted", "out_tokens", "n_emitted", "status", "accept_margin", "race_margin"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f


def test_temperature_two_is_halved_logits(oracle_mod):
    p, q, d, ua, ur = _problem(32, 64, 6, 300, 7, T=2.0)
    a = oracle_mod.verify_block(p * np.float32(0.5), q * np.float32(0.5), d, ua, ur)
    b = oracle_mod.verify_block_ex(p, q, d, ua, ur, temperature=2.0)
    for f in ("n_accepted", "out_tokens", "n_emitted", "accept_margin", "race_margin"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f
    # and it is not the T = 1 result
    c = oracle_mod.verify_block(p, q, d, ua, ur)
    assert not np.array_equal(a.accept_margin, c.accept_margin)


def _shared_problem(seed, Bn, K, V, Kp, T):
    """One set of distributions for every sequence; drafts drawn by numpy
    from softmax(l_q / T)."""
    rng = np.random.default_rng(seed)
    lp = (rng.standard_normal((Kp, V)) * 1.5).astype(np.float32)
    lq = (lp[:K] + rng.standard_normal((K, V))).astype(np.float32)
    P, Q = _softmax(lp / T), _softmax(lq / T)
    d = np.stack([rng.choice(V, size=Bn, p=Q[i]) for i in range(K)], axis=1).astype(np.int32)
    p = np.broadcast_to(lp, (Bn, Kp, V)).copy()
    q = np.broadcast_to(lq, (Bn, K, V)).copy()
    return p, q, d, rng, P, Q


@pytest.mark.parametrize("T,resample", [(0.6, "race"), (1.7, "race"), (1.0, "inverse_cdf"),
                                        (0.8, "inverse_cdf")])
def test_lossless_at_temperature(oracle_mod, T, resample):
    """Token i, given that it was emitted, follows softmax(l_p / T); the
    token drawn at the first rejection follows max(0, p - q) normalised."""
    Bn, K, V, Kp = 200_000, 3, 8, 4
    p, q, d, rng, P, Q = _shared_problem(77, Bn, K, V, Kp, T)
    ur = _u_race(rng, (Bn, V)) if resample == "race" else _u_accept(rng, (Bn,))
    r = oracle_mod.verify_block_ex(p, q, d, _u_accept(rng, (Bn, K)), ur, temperature=T,
                                   resample=resample)
    assert (r.status == 0).all()
    for i in range(Kp):
        sel = r.n_emitted > i
        obs = np.bincount(r.out_tokens[sel, i], minlength=V)
        res = stats.chisquare(obs, P[i] * sel.sum())
        assert res.pvalue > 1e-3, (i, res)
    for i in range(K):
        sel = r.n_accepted == i
        res_p = np.maximum(P[i] - Q[i], 0.0)
        res_p /= res_p.sum()
        obs = np.bincount(r.out_tokens[sel, i], minlength=V)
        support = res_p > 0
        assert obs[~support].sum() == 0
        res = stats.chisquare(obs[support], res_p[support] * sel.sum())
        assert res.pvalue > 1e-3, (i, res)


@pytest.mark.parametrize("T", [0.0, -1.0, float("inf"), float("nan")])
def test_invalid_temperature(oracle_mod, T):
    p, q, d, ua, ur = _problem(33, 2, 2, 16, 2)
    with pytest.raises(RuntimeError):
        oracle_mod.verify_block_ex(p, q, d, ua, ur, temperature=T)
