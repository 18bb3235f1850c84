"""Pins of the fp64 oracle of the tree sampler's verification ("Unlocking
Lossless Speedups in LLMs via Discrete Diffusion", aifromscratch.in, section
"The Psi-Spec Sampler": several candidates per position, verified in a prefix
tree, the AR distribution kept exactly).  Reading: every drafted node is a
point-mass draft, tested against the current residual in rank order.

Pins, none of which re-types the oracle's procedure:
  * a hand-worked golden example (tests/golden/tree_tiny.txt);
  * a chain tree is the linear verifier with one-hot draft distributions,
    output for output (the pinned verifier oracle, bonus row included);
  * losslessness: the first emitted token follows p at the root, the second,
    given the first, follows p at that node (chi-square, numpy-built trees);
  * a repeated sibling token is never accepted twice; malformed trees get status 1.
"""
import numpy as np
from scipy import stats

from conftest import read_golden

TWO24 = float(1 << 24)


def _ua(rng, shape):
    return (rng.integers(0, 1 << 24, size=shape) / TWO24).astype(np.float32)


def _ur(rng, shape):
    return (rng.integers(1, 1 << 24, size=shape) / TWO24).astype(np.float32)


def _softmax(l):
    e = np.exp(l - l.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def test_golden_tree_tiny(oracle_mod):
    g = read_golden("tree_tiny.txt")
    lg = np.log(np.array([g["p0"], g["p1"], g["p2"]], np.float64)).astype(np.float32)[None]
    par = np.array(g["parent"], np.int32)[None]
    tok = np.array(g["token"], np.int32)[None]
    ur = np.array(g["u_resample"], np.float32)[None]
    r = oracle_mod.tree_verify(lg, par, tok, np.array(g["u_accept"], np.float32)[None], ur)
    assert r.out_tokens[0].tolist()[:2] == [int(t) for t in g["tokens"]]
    assert r.n_accepted[0] == 1 and r.n_emitted[0] == 2 and r.path[0].tolist()[0] == 2
    r = oracle_mod.tree_verify(lg, par, tok, np.array(g["u_accept_b"], np.float32)[None], ur)
    assert r.out_tokens[0].tolist()[0] == int(g["tokens_b"][0])
    assert r.n_accepted[0] == 0 and r.n_emitted[0] == 1


def test_chain_is_the_linear_verifier_with_one_hot_drafts(oracle_mod):
    rng = np.random.default_rng(41)
    Bn, K, V = 200, 6, 50
    lp = (rng.standard_normal((Bn, K + 1, V)) * 4).astype(np.float32)
    P = _softmax(lp.astype(np.float64))
    # mostly the most likely token (long accepted runs, bonus rows), sometimes any token
    draft = np.array([[int(np.argmax(P[b, i])) if rng.random() < 0.9 else rng.integers(V)
                       for i in range(K)] for b in range(Bn)], np.int32)
    q = np.full((Bn, K, V), -np.inf, np.float32)
    for b in range(Bn):
        q[b, np.arange(K), draft[b]] = 0.0
    ua = _ua(rng, (Bn, K))
    ur = _ur(rng, (Bn, V))
    lin = oracle_mod.verify_block(lp, q, draft, ua, ur)
    par = np.tile(np.arange(-1, K, dtype=np.int32), (Bn, 1))
    tok = np.concatenate([np.zeros((Bn, 1), np.int32), draft], axis=1)
    ua_t = np.concatenate([np.zeros((Bn, 1), np.float32), ua], axis=1)
    tr = oracle_mod.tree_verify(lp, par, tok, ua_t, ur)
    assert np.array_equal(tr.n_accepted, lin.n_accepted)
    assert np.array_equal(tr.n_emitted, lin.n_emitted)
    assert np.array_equal(tr.out_tokens, lin.out_tokens)
    assert np.array_equal(tr.accept_margin[:, 1:], lin.accept_margin)
    assert np.array_equal(tr.race_margin, lin.race_margin)
    assert (tr.n_accepted < K).any() and (tr.n_accepted == K).any()


def test_lossless_two_levels(oracle_mod):
    """Root with 3 ranked candidates, each with 2 children: the first token
    follows p at the root, the second follows p at the accepted node."""
    rng = np.random.default_rng(5)
    Bn, V = 300_000, 8
    # nodes: 0 root; 1..3 children of 0; 4..9 children of 1..3 (two each)
    par = np.array([-1, 0, 0, 0, 1, 1, 2, 2, 3, 3], np.int32)
    N1 = par.size
    lg = (rng.standard_normal((N1, V)) * 1.5).astype(np.float32)
    P = _softmax(lg.astype(np.float64))
    tok = np.zeros(N1, np.int32)
    tok[1:4] = np.argsort(-P[0])[:3]                  # top 3 at the root
    for c, kids in ((1, (4, 5)), (2, (6, 7)), (3, (8, 9))):
        tok[list(kids)] = np.argsort(-P[c])[:2]
    r = oracle_mod.tree_verify(np.broadcast_to(lg, (Bn, N1, V)).copy(),
                               np.broadcast_to(par, (Bn, N1)).copy(),
                               np.broadcast_to(tok, (Bn, N1)).copy(), _ua(rng, (Bn, N1)),
                               _ur(rng, (Bn, V)))
    assert (r.status == 0).all()
    first = r.out_tokens[:, 0]
    assert stats.chisquare(np.bincount(first, minlength=V), P[0] * Bn).pvalue > 1e-3
    for c in (1, 2, 3):
        sel = r.path[:, 0] == c
        assert np.array_equal(sel, first == tok[c])    # a candidate's token is emitted only by accepting it
        obs = np.bincount(r.out_tokens[sel, 1], minlength=V)
        assert stats.chisquare(obs, P[c] * sel.sum()).pvalue > 1e-3, c


def test_repeated_sibling_and_bad_trees(oracle_mod):
    rng = np.random.default_rng(6)
    V = 5
    lg = np.log(np.array([[0.4, 0.3, 0.1, 0.1, 0.1]] * 3, np.float64)).astype(np.float32)[None]
    par = np.array([[-1, 0, 0]], np.int32)
    tok = np.array([[0, 2, 2]], np.int32)
    # node 1 (token 2) rejected, then node 2 has the same token: its residual weight is 0
    r = oracle_mod.tree_verify(lg, par, tok, np.array([[0, 0.5, 0.0]], np.float32), _ur(rng, (1, V)))
    assert r.n_accepted[0] == 0 and r.out_tokens[0, 0] != 2
    for bad_par, bad_tok in (([-1, 1, 0], [0, 1, 2]), ([0, 0, 0], [0, 1, 2]), ([-1, 0, 0], [0, 1, 5])):
        r = oracle_mod.tree_verify(lg, np.array([bad_par], np.int32), np.array([bad_tok], np.int32),
                                   np.zeros((1, 3), np.float32), _ur(rng, (1, V)))
        assert r.status[0] == 1 and r.n_emitted[0] == 0
