"""GPU parity of the LM head feeding the block verifier (logits = h . W^T,
then the verifier) against the fp64 oracle oracle_lm_head_verify_f64, in all
three strategies: the logits stored and verified, the verifier's statistics
in the GEMM's epilogue with the logits stored, and the statistics with only
the resampled rows recomputed ("Unlocking Lossless Speedups in LLMs via
Discrete Diffusion", aifromscratch.in, "The Psi-Spec Sampler"; aiany.app
summary, "Key Findings": one forward pass of the AR model verifies the block).
Accepted lengths, tokens and statuses are bit-exact outside fp64 near-ties
(margin < 1e-4), which must stay under 0.1% of sequences."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import compare_verify, require_gpu
from lossless_draft_verify_gated_b300 import inputs

pytestmark = pytest.mark.gpu

MODES = ["plain", "stats_store", "stats_recompute"]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _drafts(pr):
    """Drafts drawn from the draft rows' logits (fp64 matmul of the bf16
    values, rounded to fp32) by the oracle's sampler."""
    Bn, K, Kp = pr.Bn, pr.K, pr.Kp
    hq = pr.h[Bn * Kp:].double()
    lq = (hq @ pr.W.double().T).float().reshape(Bn, K, -1)
    d, st, _ = oracle.draft_sample(lq, pr.u_draft)
    assert (st == 0).all()
    return d.reshape(Bn, K)


def _oracle(pr, draft):
    Bn, K, Kp = pr.Bn, pr.K, pr.Kp
    d = pr.h.shape[1]
    h = pr.h.double().numpy()
    W = pr.W.double().numpy()  # one head for both pathways
    return oracle.lm_head_verify(h[:Bn * Kp].reshape(Bn, Kp, d), h[Bn * Kp:].reshape(Bn, K, d),
                                 W, W, draft, pr.u_accept, pr.u_resample)


def _gpu(pr, draft, mode):
    from lossless_draft_verify_gated_b300 import uno_device_error, uno_lm_head_verify
    dv = "cuda"
    out = uno_lm_head_verify(pr.h.to(dv), pr.W.to(dv), torch.from_numpy(draft).to(dv),
                             pr.u_accept.to(dv), pr.u_resample.to(dv), Kp=pr.Kp, mode=mode)
    torch.cuda.synchronize()
    assert uno_device_error() == 0
    return out


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("Bn,K,V,d,Kp", [(2, 4, 1000, 256, None), (3, 5, 4104, 512, 6),
                                          (70, 4, 2048, 256, None), (9, 16, 8192, 1024, 17),
                                          (6, 12, 4096, 512, 13)])  # 150 rows: just above the weights-as-A limit
def test_lm_head_parity(mode, Bn, K, V, d, Kp):
    pr = inputs.lm_head_problem(Bn, K, V, d, Kp=Kp, sigma=1.0)
    draft = _drafts(pr)
    ref = _oracle(pr, draft)
    compare_verify(_gpu(pr, draft, mode), ref, Bn)
    assert ref.n_emitted.sum() >= Bn


@pytest.mark.parametrize("Bn", [1, 16])
def test_lm_head_full_size(Bn):
    """Llama-3-8B head shape (d 4096, vocab 128256), block 16, every strategy
    against the oracle on the same inputs."""
    pr = inputs.lm_head_problem(Bn, 16, 128256, 4096, sigma=1.0)
    draft = _drafts(pr)
    ref = _oracle(pr, draft)
    for mode in MODES + ["auto"]:
        compare_verify(_gpu(pr, draft, mode), ref, Bn)


def test_lm_head_status_codes():
    pr = inputs.lm_head_problem(4, 3, 512, 128)
    draft = _drafts(pr)
    draft[1, 2] = 512          # outside the vocabulary
    draft[2, 0] = -1
    h = pr.h.clone()
    h[3 * pr.Kp + 1, 5] = float("nan")  # an AR row of sequence 3 (rows b*Kp + j)
    pr2 = inputs.LmHeadProblem(h, pr.W, pr.u_accept, pr.u_resample, pr.u_draft, pr.Bn, pr.K, pr.Kp)
    ref = _oracle(pr2, draft)
    for mode in MODES:
        out = _gpu(pr2, draft, mode)
        compare_verify(out, ref, 4)
        assert out[3].cpu().tolist() == [0, 1, 1, 2]
