"""GPU parity of the block verifier and the draft sampler against the fp64
oracle, on seeded inputs: bit-exact accepted lengths, emitted tokens and
statuses outside fp64 near-ties (margin < 1e-4), which must stay under 0.1%.
("Unlocking Lossless Speedups in LLMs via Discrete Diffusion",
aifromscratch.in, section "The Psi-Spec Sampler".)"""
import numpy as np
import pytest
import torch
from scipy import stats

import oracle
from gpu_util import compare_verify, require_gpu
from lossless_draft_verify_gated_b300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _run_case(Bn, K, V, Kp=None, sigma=1.0, seed=inputs.BASE_SEED):
    from lossless_draft_verify_gated_b300 import uno_verify_block
    pr = inputs.verify_problem(Bn, K, V, Kp=Kp, sigma=sigma, seed=seed)
    draft, st, _ = oracle.draft_sample(pr.q_logits, pr.u_draft)
    assert (st == 0).all()
    draft = draft.reshape(Bn, K)
    ref = oracle.verify_block(pr.p_logits, pr.q_logits, draft, pr.u_accept, pr.u_resample)
    dev = "cuda"
    gpu = uno_verify_block(pr.p_logits.to(dev), pr.q_logits.to(dev),
                           torch.from_numpy(draft).to(dev), pr.u_accept.to(dev),
                           pr.u_resample.to(dev))
    torch.cuda.synchronize()
    ties = compare_verify(gpu, ref, Bn)
    return ref, gpu, ties


@pytest.mark.parametrize("Bn,K,V,Kp,sigma", [
    (2, 4, 1000, None, 1.0),      # the tiny smoke configuration
    (13, 4, 999, 5, 1.0),         # ragged vocab (rows not 16-byte aligned) and a bonus row
    (7, 16, 128256, None, 0.25),  # full vocab, high acceptance
    (7, 16, 128256, 17, 1.0),     # full vocab with bonus row
    (5, 3, 3, None, 4.0),         # vocab smaller than a warp
    (64, 16, 4099, None, 4.0),    # low acceptance, odd vocab
    (1, 1, 1, 2, 1.0),            # a one-token vocabulary
])
def test_verify_parity(Bn, K, V, Kp, sigma):
    _run_case(Bn, K, V, Kp, sigma)


@pytest.mark.parametrize("sigma", [0.25, 1.0, 4.0])
def test_verify_parity_full_size(sigma):
    """batch 256 x block 16 x vocab 128256, the verifier's full configuration."""
    ref, gpu, ties = _run_case(256, 16, 128256, None, sigma)
    mean_em = gpu[2].float().mean().item()
    assert mean_em >= 1.0


@pytest.mark.parametrize("Bn", [1, 8, 32, 128, 512])
def test_verify_parity_step_sweep(Bn):
    """The verifier of the benchmarked step at every batch of the sweep
    (block 16, vocab 128256, sigma 1), each with its own launch plan (at batch
    1 the statistics pass splits every row 37 ways and the race 126 ways);
    every sequence against the oracle."""
    ref, gpu, ties = _run_case(Bn, 16, 128256, None, 1.0)
    assert gpu[2].sum().item() >= Bn


def _shifted(t):
    """A contiguous copy of t whose data start 4 bytes past a 16-byte boundary
    (rows stay 4-byte aligned): the statistics pass then reads every row
    through its scalar head and tail."""
    buf = torch.empty(t.numel() + 4, dtype=t.dtype, device=t.device)
    v = buf[1:1 + t.numel()].view(t.shape)
    v.copy_(t)
    assert v.data_ptr() % 16 == 4
    return v


@pytest.mark.parametrize("Bn,K,V,Kp", [(1, 16, 128256, None), (3, 16, 128256, 17),
                                       (16, 16, 128256, None), (5, 7, 1000, 8), (16, 4, 64, None)])
def test_aligned_and_unaligned_rows(Bn, K, V, Kp):
    """The same inputs from 16-byte aligned rows and from rows 4 bytes off
    alignment (the vectorised statistics pass's head/tail path) match the
    oracle and each other, at batches on both sides of the finish kernel's
    programmatic-launch threshold."""
    from lossless_draft_verify_gated_b300 import uno_device_error, uno_verify_block
    pr = inputs.verify_problem(Bn, K, V, Kp=Kp, sigma=1.0, seed=77)
    draft, st, _ = oracle.draft_sample(pr.q_logits, pr.u_draft)
    draft = draft.reshape(Bn, K)
    ref = oracle.verify_block(pr.p_logits, pr.q_logits, draft, pr.u_accept, pr.u_resample)
    args = [pr.p_logits.cuda(), pr.q_logits.cuda(), torch.from_numpy(draft).cuda(),
            pr.u_accept.cuda(), pr.u_resample.cuda()]
    one = uno_verify_block(*args)
    two = uno_verify_block(_shifted(args[0]), _shifted(args[1]), args[2], args[3], _shifted(args[4]))
    torch.cuda.synchronize()
    compare_verify(one, ref, Bn)
    compare_verify(two, ref, Bn)
    assert uno_device_error() == 0


def test_q_equals_p_accepts_all():
    from lossless_draft_verify_gated_b300 import uno_verify_block
    Bn, K, V = 33, 8, 5000
    pr = inputs.verify_problem(Bn, K, V, Kp=K + 1)
    q = pr.p_logits[:, :K].contiguous()
    draft = torch.randint(0, V, (Bn, K), dtype=torch.int32, generator=inputs.generator("qp"))
    n_acc, toks, n_em, st = uno_verify_block(pr.p_logits.cuda(), q.cuda(), draft.cuda(),
                                             pr.u_accept.cuda(), pr.u_resample.cuda())
    assert (n_acc.cpu() == K).all() and (n_em.cpu() == K + 1).all() and (st.cpu() == 0).all()
    assert torch.equal(toks[:, :K].cpu(), draft)


def test_status_codes_and_empty():
    from lossless_draft_verify_gated_b300 import uno_verify_block
    Bn, K, V = 5, 2, 64
    pr = inputs.verify_problem(Bn, K, V)
    p, q = pr.p_logits.clone(), pr.q_logits.clone()
    draft = torch.randint(0, V, (Bn, K), dtype=torch.int32, generator=inputs.generator("st"))
    draft[1, 1] = V
    draft[2, 0] = -7
    p[3, 1, 5] = float("nan")
    q[4, 0, :] = float("-inf")
    p[0, 0, 3] = float("-inf")
    ref = oracle.verify_block(p, q, draft, pr.u_accept, pr.u_resample)
    gpu = uno_verify_block(p.cuda(), q.cuda(), draft.cuda(), pr.u_accept.cuda(), pr.u_resample.cuda())
    compare_verify(gpu, ref, Bn)
    assert gpu[3].cpu().tolist() == [0, 1, 1, 2, 2]
    e = torch.empty(0, device="cuda")
    out = uno_verify_block(e.reshape(0, 2, 4), e.reshape(0, 2, 4), torch.empty(0, 2, dtype=torch.int32,
                           device="cuda"), e.reshape(0, 2), e.reshape(0, 4))
    assert out[0].numel() == 0


def test_gpu_losslessness_chi_square():
    """10^6 sequences, vocab 8, block 3 + bonus: every emitted position is
    distributed as p_i (the losslessness invariant), measured on the GPU."""
    from lossless_draft_verify_gated_b300 import uno_draft_sample, uno_verify_block
    Bn, K, V = 1_000_000, 3, 8
    g = inputs.generator("chi")
    lp = torch.randn(K + 1, V, generator=g) * 1.5
    lq = lp[:K] + torch.randn(K, V, generator=g)
    p = lp.expand(Bn, K + 1, V).contiguous().cuda()
    q = lq.expand(Bn, K, V).contiguous().cuda()
    ud = inputs.uniform_race((Bn, K, V), "chi.ud").cuda()
    draft, st = uno_draft_sample(q, ud)
    assert (st == 0).all()
    ua = inputs.uniform_accept((Bn, K), "chi.ua").cuda()
    ur = inputs.uniform_race((Bn, V), "chi.ur").cuda()
    n_acc, toks, n_em, st = uno_verify_block(p, q, draft, ua, ur)
    toks, n_em = toks.cpu().numpy(), n_em.cpu().numpy()
    P = torch.softmax(lp.double(), -1).numpy()
    for i in range(K + 1):
        sel = n_em > i
        obs = np.bincount(toks[sel, i], minlength=V)
        res = stats.chisquare(obs, P[i] * sel.sum())
        assert res.pvalue > 1e-3, (i, res)
    Q = torch.softmax(lq.double(), -1).numpy()
    obs = np.bincount(draft[:, 0].cpu().numpy(), minlength=V)
    assert stats.chisquare(obs, Q[0] * Bn).pvalue > 1e-3


@pytest.mark.parametrize("R,V", [(64, 128256), (1000, 7), (5, 1), (33, 4097)])
def test_draft_sample_parity(R, V):
    from lossless_draft_verify_gated_b300 import uno_draft_sample
    lg = inputs.normal((R, V), 3.0, f"ds.l.{R}.{V}")
    u = inputs.uniform_race((R, V), f"ds.u.{R}.{V}")
    ref_tok, ref_st, margin = oracle.draft_sample(lg, u)
    tok, st = uno_draft_sample(lg.cuda(), u.cuda())
    tok, st = tok.cpu().numpy(), st.cpu().numpy()
    keep = margin >= 1e-4
    np.testing.assert_array_equal(st, ref_st)
    np.testing.assert_array_equal(tok[keep], ref_tok[keep])
    assert (~keep).sum() <= max(1, R // 1000)
