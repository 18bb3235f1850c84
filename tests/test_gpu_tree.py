"""GPU parity of the tree sampler's verification against the fp64 oracle
("Unlocking Lossless Speedups in LLMs via Discrete Diffusion",
aifromscratch.in, section "The Psi-Spec Sampler": the top K candidates of each
position, verified in a prefix tree, the AR distribution kept).  Accepted
depths, paths, emitted tokens and statuses are bit-exact outside fp64
near-ties (an accept test or the race with margin < 1e-4), which must stay
under 0.1% of sequences; losslessness is checked on the GPU by chi-square."""
import numpy as np
import pytest
import torch
from scipy import stats

import oracle
from gpu_util import MAX_NEAR_TIE_FRAC, NEAR_TIE, require_gpu
from lossless_draft_verify_gated_b300 import inputs

pytestmark = pytest.mark.gpu

TWO24 = float(1 << 24)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _ua(rng, shape):
    return (rng.integers(0, 1 << 24, size=shape) / TWO24).astype(np.float32)


def _ur(rng, shape):
    return (rng.integers(1, 1 << 24, size=shape) / TWO24).astype(np.float32)


def _topk_tree(lg, widths, rng=None):
    """A tree whose children at each node are the most likely tokens of that
    node's row (the top-k drafting of the tree sampler); widths[d] children per
    node at depth d.  Returns parent, token [N+1]."""
    parent, token, depth = [-1], [0], [0]
    frontier = [0]
    for w in widths:
        nxt = []
        for node in frontier:
            top = np.argsort(-lg[node])[:w]
            for t in top:
                if len(parent) >= lg.shape[0]:
                    break
                parent.append(node)
                token.append(int(t))
                nxt.append(len(parent) - 1)
        frontier = nxt
    n1 = len(parent)
    return np.array(parent, np.int32), np.array(token, np.int32), n1


def _compare(gpu, ref, Bn):
    n_acc, pth, toks, n_em, st = (t.cpu().numpy() for t in gpu)
    tie = (ref.accept_margin < NEAR_TIE).any(axis=1) | (ref.race_margin < NEAR_TIE)
    keep = ~tie
    np.testing.assert_array_equal(st, ref.status)
    np.testing.assert_array_equal(n_acc[keep], ref.n_accepted[keep])
    np.testing.assert_array_equal(n_em[keep], ref.n_emitted[keep])
    np.testing.assert_array_equal(toks[keep], ref.out_tokens[keep])
    if pth.size:
        np.testing.assert_array_equal(pth[keep], ref.path[keep])
    assert tie.sum() <= max(1, MAX_NEAR_TIE_FRAC * Bn), f"{tie.sum()} near ties of {Bn}"
    return int(tie.sum())


def _run(lg, par, tok, ua, ur):
    from lossless_draft_verify_gated_b300 import uno_tree_verify
    ref = oracle.tree_verify(lg, par, tok, ua, ur)
    d = "cuda"
    gpu = uno_tree_verify(torch.from_numpy(lg).to(d), torch.from_numpy(par).to(d),
                          torch.from_numpy(tok).to(d), torch.from_numpy(ua).to(d),
                          torch.from_numpy(ur).to(d))
    torch.cuda.synchronize()
    return ref, gpu


@pytest.mark.parametrize("Bn,N,V", [(4, 16, 128256), (9, 5, 999), (40, 7, 64)])
def test_chain_trees(Bn, N, V):
    """Chains (one candidate per position, mostly the most likely token)."""
    rng = np.random.default_rng(N * 1000 + V)
    # peaked rows at a large vocabulary, so that the most likely token is often accepted
    lg = (rng.standard_normal((Bn, N + 1, V)) * (8 if V > 10000 else 3)).astype(np.float32)
    par = np.tile(np.arange(-1, N, dtype=np.int32), (Bn, 1))
    tok = np.zeros((Bn, N + 1), np.int32)
    for b in range(Bn):
        for j in range(1, N + 1):
            tok[b, j] = np.argmax(lg[b, j - 1]) if rng.random() < 0.8 else rng.integers(V)
    ref, gpu = _run(lg, par, tok, _ua(rng, (Bn, N + 1)), _ur(rng, (Bn, V)))
    _compare(gpu, ref, Bn)
    assert (ref.n_accepted > 0).any()


@pytest.mark.parametrize("Bn,widths,V", [(6, (3, 2, 2, 1), 128256), (16, (4, 2, 1), 4099),
                                        (3, (8, 4), 1000)])
def test_topk_trees(Bn, widths, V):
    """Bushy trees whose children are each node's most likely tokens."""
    rng = np.random.default_rng(len(widths) * 7 + V)
    n1 = 1
    for w in np.cumprod(widths):
        n1 += int(w)
    lg = (rng.standard_normal((Bn, n1, V)) * (8 if V > 10000 else 6)).astype(np.float32)
    par = np.zeros((Bn, n1), np.int32)
    tok = np.zeros((Bn, n1), np.int32)
    for b in range(Bn):
        p_, t_, m = _topk_tree(lg[b], widths)
        assert m == n1
        par[b], tok[b] = p_, t_
    ref, gpu = _run(lg, par, tok, _ua(rng, (Bn, n1)), _ur(rng, (Bn, V)))
    _compare(gpu, ref, Bn)
    assert (ref.n_accepted >= 2).any()


def test_random_trees_and_repeated_tokens():
    """Random shapes (parent uniform below the node), random tokens from a small
    set so that siblings repeat, vocabulary of 37."""
    rng = np.random.default_rng(3)
    Bn, N, V = 300, 24, 37
    lg = (rng.standard_normal((Bn, N + 1, V)) * 1.5).astype(np.float32)
    par = np.zeros((Bn, N + 1), np.int32)
    par[:, 0] = -1
    for j in range(1, N + 1):
        par[:, j] = rng.integers(0, j, size=Bn)
    tok = rng.integers(0, 6, size=(Bn, N + 1)).astype(np.int32)
    ref, gpu = _run(lg, par, tok, _ua(rng, (Bn, N + 1)), _ur(rng, (Bn, V)))
    _compare(gpu, ref, Bn)


def test_root_only_and_status_codes():
    rng = np.random.default_rng(11)
    V = 50
    # N = 0: plain sampling from p at the root
    lg = (rng.standard_normal((5, 1, V)) * 2).astype(np.float32)
    ref, gpu = _run(lg, np.full((5, 1), -1, np.int32), np.zeros((5, 1), np.int32),
                    _ua(rng, (5, 1)), _ur(rng, (5, V)))
    _compare(gpu, ref, 5)
    assert (gpu[3].cpu() == 1).all()
    # malformed trees, and a non-finite row on / off the walked path
    Bn, N = 6, 3
    lg = (rng.standard_normal((Bn, N + 1, V))).astype(np.float32)
    par = np.tile(np.array([-1, 0, 0, 1], np.int32), (Bn, 1))
    tok = np.tile(np.array([0, 3, 4, 5], np.int32), (Bn, 1))
    par[1, 2] = 2            # parent not below the node
    tok[2, 3] = V            # token out of range
    par[3, 0] = 0            # root with a parent
    lg[4, 0, 7] = np.nan     # the root's row: always walked
    lg[5, 2, :] = -np.inf    # node 2's row: walked only if node 2 is accepted
    ua = np.zeros((Bn, N + 1), np.float32)
    ua[5, 1] = 0.999         # node 1 rejected at sequence 5 ...
    ref, gpu = _run(lg, par, tok, ua, _ur(rng, (Bn, V)))
    _compare(gpu, ref, Bn)
    st = gpu[4].cpu().tolist()
    assert st[1] == st[2] == st[3] == 1 and st[4] == 2


def test_gpu_tree_losslessness_chi_square():
    """10^6 walks of a two-level top-3 / top-2 tree at vocab 8 on the GPU: the
    first emitted token follows p at the root, the second follows p at the
    accepted node."""
    from lossless_draft_verify_gated_b300 import uno_tree_verify
    rng = np.random.default_rng(5)
    Bn, V = 1_000_000, 8
    par = np.array([-1, 0, 0, 0, 1, 1, 2, 2, 3, 3], np.int32)
    N1 = par.size
    lg = (rng.standard_normal((N1, V)) * 1.5).astype(np.float32)
    P = torch.softmax(torch.from_numpy(lg).double(), -1).numpy()
    tok = np.zeros(N1, np.int32)
    tok[1:4] = np.argsort(-lg[0])[:3]
    for c, kids in ((1, (4, 5)), (2, (6, 7)), (3, (8, 9))):
        tok[list(kids)] = np.argsort(-lg[c])[:2]
    d = "cuda"
    L = torch.from_numpy(lg).to(d).expand(Bn, N1, V).contiguous()
    Pa = torch.from_numpy(par).to(d).expand(Bn, N1).contiguous()
    T = torch.from_numpy(tok).to(d).expand(Bn, N1).contiguous()
    ua = inputs.uniform_accept((Bn, N1), "tree.chi.ua").to(d)
    ur = inputs.uniform_race((Bn, V), "tree.chi.ur").to(d)
    n_acc, pth, toks, n_em, st = uno_tree_verify(L, Pa, T, ua, ur)
    toks, pth = toks.cpu().numpy(), pth.cpu().numpy()
    assert int(st.abs().sum()) == 0
    first = toks[:, 0]
    assert stats.chisquare(np.bincount(first, minlength=V), P[0] * Bn).pvalue > 1e-3
    for c in (1, 2, 3):
        sel = pth[:, 0] == c
        assert np.array_equal(sel, first == tok[c])
        obs = np.bincount(toks[sel, 1], minlength=V)
        assert stats.chisquare(obs, P[c] * sel.sum()).pvalue > 1e-3, c


def test_chain_equals_linear_verifier_on_gpu():
    """On the GPU as in the oracle: a chain tree verifies exactly like the
    linear block verifier whose draft distributions are one-hot at the drafted
    tokens (a point-mass draft), bonus row included."""
    from lossless_draft_verify_gated_b300 import uno_tree_verify, uno_verify_block
    rng = np.random.default_rng(17)
    Bn, K, V = 64, 8, 128256
    lp = (rng.standard_normal((Bn, K + 1, V)) * 8).astype(np.float32)
    draft = np.where(rng.random((Bn, K)) < 0.85, np.argmax(lp[:, :K], axis=2),
                     rng.integers(0, V, (Bn, K))).astype(np.int32)
    q = np.full((Bn, K, V), -np.inf, np.float32)
    np.put_along_axis(q, draft[:, :, None], 0.0, axis=2)
    ua = _ua(rng, (Bn, K))
    ur = _ur(rng, (Bn, V))
    d = "cuda"
    lin = uno_verify_block(torch.from_numpy(lp).to(d), torch.from_numpy(q).to(d),
                           torch.from_numpy(draft).to(d), torch.from_numpy(ua).to(d),
                           torch.from_numpy(ur).to(d))
    par = np.tile(np.arange(-1, K, dtype=np.int32), (Bn, 1))
    tok = np.concatenate([np.zeros((Bn, 1), np.int32), draft], axis=1)
    ua_t = np.concatenate([np.zeros((Bn, 1), np.float32), ua], axis=1)
    tr = uno_tree_verify(torch.from_numpy(lp).to(d), torch.from_numpy(par).to(d),
                         torch.from_numpy(tok).to(d), torch.from_numpy(ua_t).to(d),
                         torch.from_numpy(ur).to(d))
    torch.cuda.synchronize()
    # both sides decide in fp32: compare outside the oracle's near ties
    ref = oracle.tree_verify(lp, par, tok, ua_t, ur)
    keep = ~((ref.accept_margin < NEAR_TIE).any(axis=1) | (ref.race_margin < NEAR_TIE))
    n_lin, t_lin = lin[0].cpu().numpy(), lin[1].cpu().numpy()
    n_tr, t_tr = tr[0].cpu().numpy(), tr[2].cpu().numpy()
    np.testing.assert_array_equal(n_lin[keep], n_tr[keep])
    np.testing.assert_array_equal(t_lin[keep], t_tr[keep, :K + 1])
    assert (n_lin == K).any() and (n_lin < K).any()
