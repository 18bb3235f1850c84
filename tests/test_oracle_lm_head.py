"""Pins of the fp64 oracle of the LM head feeding the verifier (logits =
h . W^T over the vocabulary, then the block verifier; "Unlocking Lossless
Speedups in LLMs via Discrete Diffusion", aifromscratch.in, section "The
Psi-Spec Sampler": the AR model verifies the drafted block in one forward
pass, whose last step is the LM head).

Pins, none of which re-types the oracle's procedure:
  * with small integer hidden states and weights in quarter steps every logit
    is exact in fp32 and fp64, so the result must equal the (pinned) verifier
    oracle run on numpy's h @ W.T, output for output -- this fixes the
    orientation of the product (W is [V, d]) and which head serves which rows;
  * the hand-worked golden example of the verifier (tests/golden/verify_tiny.txt)
    reached through a one-dimensional hidden state;
  * the draft rows use W_q: swapping the heads changes the result.
"""
import numpy as np

from conftest import read_golden

TWO24 = float(1 << 24)


def _exact_problem(seed, Bn, K, Kp, V, d):
    rng = np.random.default_rng(seed)
    hp = rng.integers(-2, 3, size=(Bn, Kp, d)).astype(np.float64)
    hq = rng.integers(-2, 3, size=(Bn, K, d)).astype(np.float64)
    Wp = rng.integers(-6, 7, size=(V, d)).astype(np.float64) / 4
    Wq = Wp + rng.integers(-2, 3, size=(V, d)).astype(np.float64) / 4
    draft = rng.integers(0, V, size=(Bn, K)).astype(np.int32)
    ua = (rng.integers(0, 1 << 24, size=(Bn, K)) / TWO24).astype(np.float32)
    ur = (rng.integers(1, 1 << 24, size=(Bn, V)) / TWO24).astype(np.float32)
    return hp, hq, Wp, Wq, draft, ua, ur


def test_equals_verifier_on_numpy_logits(oracle_mod):
    for Kp in (6, 7):
        hp, hq, Wp, Wq, draft, ua, ur = _exact_problem(5 + Kp, 40, 6, Kp, 300, 24)
        lp = np.einsum("bkd,vd->bkv", hp, Wp)
        lq = np.einsum("bkd,vd->bkv", hq, Wq)
        assert np.array_equal(lp.astype(np.float32).astype(np.float64), lp)  # exact in fp32
        a = oracle_mod.verify_block(lp.astype(np.float32), lq.astype(np.float32), draft, ua, ur)
        b = oracle_mod.lm_head_verify(hp, hq, Wp, Wq, draft, ua, ur)
        for f in ("n_accepted", "out_tokens", "n_emitted", "status", "accept_margin", "race_margin"):
            assert np.array_equal(getattr(a, f), getattr(b, f)), f
        assert (b.n_accepted < 6).any() and (b.n_emitted > b.n_accepted).any()


def test_draft_rows_use_the_draft_head(oracle_mod):
    hp, hq, Wp, Wq, draft, ua, ur = _exact_problem(21, 40, 6, 6, 300, 24)
    a = oracle_mod.lm_head_verify(hp, hq, Wp, Wq, draft, ua, ur)
    b = oracle_mod.lm_head_verify(hp, hq, Wp, Wp, draft, ua, ur)
    assert not np.array_equal(a.accept_margin, b.accept_margin)


def test_golden_verify_tiny_through_the_head(oracle_mod):
    g = read_golden("verify_tiny.txt")
    V, K = int(g["V"][0]), int(g["K"][0])
    # d = 1, h = 1: the logits are the head's single column
    Wp = np.log(np.array([g["p0"], g["p1"]], np.float64))   # [K, V]: one head per position
    Wq = np.log(np.array([g["q0"], g["q1"]], np.float64))
    d = np.array(g["draft"], np.int32)[None]
    ua = np.array(g["u_accept"], np.float32)[None]
    ur = np.array(g["u_resample"], np.float32)[None]
    # the head is shared by the positions, so put position i's logits in a
    # one-hot hidden dimension: h[i] = e_i, W[v, i] = logit_i(v)
    hp = np.eye(K)[None]
    Wp_, Wq_ = Wp.T.copy(), Wq.T.copy()                     # [V, d = K]
    r = oracle_mod.lm_head_verify(hp, hp.copy(), Wp_, Wq_, d, ua, ur)
    assert r.n_accepted[0] == g["n_accepted"][0]
    assert r.n_emitted[0] == g["n_emitted"][0]
    assert r.out_tokens[0].tolist() == [int(t) for t in g["out_tokens"]]
    assert r.status[0] == 0 and V == 3
