"""GPU parity of the verifier's sampling variants (temperature T, single-
uniform inverse-CDF resample) against the fp64 oracle.  ("Unlocking Lossless
Speedups in LLMs via Discrete Diffusion", aifromscratch.in, section "The
Psi-Spec Sampler": the speculative-decoding acceptance rule, every
distribution taken at temperature T.)

The race at any T is compared bit-exact outside fp64 near-ties, as the plain
verifier.  The inverse CDF picks the bucket that holds u * S; the kernel's
fp32 weights (summed exactly in fixed point) move bucket edges by about 2e-7 of S, so its
token is compared where the oracle's edge margin is at least 1e-6 of S, and
its distribution is checked by chi-square."""
import numpy as np
import pytest
import torch
from scipy import stats

import oracle
from gpu_util import compare_verify, require_gpu
from lossless_draft_verify_gated_b300 import inputs

pytestmark = pytest.mark.gpu

EDGE_TOL = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _drafts_at(q_logits, u_draft, T):
    """Drafts drawn from softmax(l_q / T) by the oracle's race (inputs, not outputs)."""
    scaled = (q_logits.double() / T).float()
    d, st, _ = oracle.draft_sample(scaled, u_draft)
    assert (st == 0).all()
    return d.reshape(q_logits.shape[0], q_logits.shape[1])


def _gpu_ex(pr, draft, ur, T, resample):
    from lossless_draft_verify_gated_b300 import uno_verify_block_ex
    out = uno_verify_block_ex(pr.p_logits.cuda(), pr.q_logits.cuda(), torch.from_numpy(draft).cuda(),
                              pr.u_accept.cuda(), ur.cuda(), temperature=T, resample=resample)
    torch.cuda.synchronize()
    return out


def test_unit_temperature_race_equals_plain_verifier():
    from lossless_draft_verify_gated_b300 import uno_verify_block
    Bn, K, V = 16, 16, 128256
    pr = inputs.verify_problem(Bn, K, V, Kp=K + 1)
    draft = _drafts_at(pr.q_logits, pr.u_draft, 1.0)
    a = uno_verify_block(pr.p_logits.cuda(), pr.q_logits.cuda(), torch.from_numpy(draft).cuda(),
                         pr.u_accept.cuda(), pr.u_resample.cuda())
    b = _gpu_ex(pr, draft, pr.u_resample, 1.0, "race")
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("Bn,K,V,Kp,T", [
    (8, 16, 128256, None, 0.5),
    (8, 16, 128256, 17, 2.0),
    (13, 4, 999, 5, 0.7),
    (64, 16, 4099, None, 1.3),
])
def test_race_at_temperature_parity(Bn, K, V, Kp, T):
    pr = inputs.verify_problem(Bn, K, V, Kp=Kp)
    draft = _drafts_at(pr.q_logits, pr.u_draft, T)
    ref = oracle.verify_block_ex(pr.p_logits, pr.q_logits, draft, pr.u_accept, pr.u_resample,
                                 temperature=T, resample="race")
    gpu = _gpu_ex(pr, draft, pr.u_resample, T, "race")
    compare_verify(gpu, ref, Bn)


def _u_single(Bn, name):
    return inputs.uniform_accept((Bn,), name)


@pytest.mark.parametrize("Bn,K,V,Kp,T,sigma", [
    (32, 16, 128256, None, 1.0, 1.0),
    (16, 16, 128256, 17, 0.8, 0.25),
    (64, 16, 4099, None, 1.0, 4.0),
    (13, 4, 999, 5, 1.5, 1.0),
    (5, 3, 3, None, 1.0, 4.0),
])
def test_inverse_cdf_parity(Bn, K, V, Kp, T, sigma):
    pr = inputs.verify_problem(Bn, K, V, Kp=Kp, sigma=sigma)
    draft = _drafts_at(pr.q_logits, pr.u_draft, T)
    u1 = _u_single(Bn, f"icdf.{Bn}.{V}")
    ref = oracle.verify_block_ex(pr.p_logits, pr.q_logits, draft, pr.u_accept, u1,
                                 temperature=T, resample="inverse_cdf")
    n_acc, toks, n_em, st = (t.cpu().numpy() for t in _gpu_ex(pr, draft, u1, T, "inverse_cdf"))
    np.testing.assert_array_equal(st, ref.status)
    acc_tie = (ref.accept_margin < 1e-4).any(axis=1)
    keep = ~acc_tie
    np.testing.assert_array_equal(n_acc[keep], ref.n_accepted[keep])
    np.testing.assert_array_equal(n_em[keep], ref.n_emitted[keep])
    edge = ref.race_margin < EDGE_TOL
    same = keep & ~edge
    np.testing.assert_array_equal(toks[same], ref.out_tokens[same])
    assert acc_tie.mean() <= 0.02 and edge.mean() <= 0.05, (acc_tie.sum(), edge.sum())
    drawn = keep & (n_em > n_acc)
    assert drawn.any()


def test_inverse_cdf_chi_square():
    """10^6 sequences, vocab 8, block 3 + bonus, T = 0.8: the token drawn at
    the first rejection follows max(0, p - q)/S and every emitted position
    follows p, measured on the GPU."""
    from lossless_draft_verify_gated_b300 import uno_draft_sample, uno_verify_block_ex
    Bn, K, V, T = 1_000_000, 3, 8, 0.8
    g = inputs.generator("icdf.chi")
    lp = torch.randn(K + 1, V, generator=g) * 1.5
    lq = lp[:K] + torch.randn(K, V, generator=g)
    p = lp.expand(Bn, K + 1, V).contiguous().cuda()
    q = lq.expand(Bn, K, V).contiguous().cuda()
    ud = inputs.uniform_race((Bn, K, V), "icdf.chi.ud").cuda()
    draft, st = uno_draft_sample((q.double() / T).float(), ud)
    assert (st == 0).all()
    ua = inputs.uniform_accept((Bn, K), "icdf.chi.ua").cuda()
    u1 = inputs.uniform_accept((Bn,), "icdf.chi.u1").cuda()
    n_acc, toks, n_em, st = uno_verify_block_ex(p, q, draft, ua, u1, temperature=T,
                                                resample="inverse_cdf")
    n_acc, toks, n_em = n_acc.cpu().numpy(), toks.cpu().numpy(), n_em.cpu().numpy()
    P = torch.softmax(lp.double() / T, -1).numpy()
    Q = torch.softmax(lq.double() / T, -1).numpy()
    for i in range(K + 1):
        sel = n_em > i
        res = stats.chisquare(np.bincount(toks[sel, i], minlength=V), P[i] * sel.sum())
        assert res.pvalue > 1e-3, (i, res)
    for i in range(K):
        sel = n_acc == i
        r = np.maximum(P[i] - Q[i], 0.0)
        r /= r.sum()
        obs = np.bincount(toks[sel, i], minlength=V)
        assert obs[r == 0].sum() == 0
        res = stats.chisquare(obs[r > 0], r[r > 0] * sel.sum())
        assert res.pvalue > 1e-3, (i, res)


@pytest.mark.parametrize("T", [0.0, -2.0, float("inf"), float("nan")])
def test_bad_temperature_rejected(T):
    from lossless_draft_verify_gated_b300 import UnoError, uno_verify_block_ex
    pr = inputs.verify_problem(2, 2, 64)
    draft = torch.zeros((2, 2), dtype=torch.int32).cuda()
    with pytest.raises(UnoError):
        uno_verify_block_ex(pr.p_logits.cuda(), pr.q_logits.cuda(), draft, pr.u_accept.cuda(),
                            pr.u_resample.cuda(), temperature=T)


def test_unknown_mode_rejected():
    from lossless_draft_verify_gated_b300 import lib
    rc = lib().uno_verify_block_ex(None, None, None, None, None, 1, 1, 1, 8, 1.0, 7,
                                   None, None, None, None, None, 0, None)
    assert rc == -1  # UNO_ERR_ARG
