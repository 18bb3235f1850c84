"""Helpers shared by the GPU parity tests (no method arithmetic here)."""
import numpy as np
import pytest
import torch

NEAR_TIE = 1e-4          # fp64 decision margin below which a sequence is excluded
MAX_NEAR_TIE_FRAC = 1e-3  # at most 0.1% of sequences may be excluded
GEMM_TOL = 2e-2          # max |y_gpu - y_ref| <= GEMM_TOL * rms(y_ref)


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lossless_draft_verify_gated_b300 import build
    build.build()


def compare_verify(gpu, ref, n_seq):
    """Bit-exact comparison of the verifier outputs outside fp64 near-ties.
    gpu = (n_acc, toks, n_em, status) torch tensors; ref = oracle.VerifyResult."""
    n_acc, toks, n_em, st = (t.cpu().numpy() for t in gpu)
    tie = ref.near_tie(NEAR_TIE)
    keep = ~tie
    np.testing.assert_array_equal(st, ref.status)
    np.testing.assert_array_equal(n_acc[keep], ref.n_accepted[keep])
    np.testing.assert_array_equal(n_em[keep], ref.n_emitted[keep])
    np.testing.assert_array_equal(toks[keep], ref.out_tokens[keep])
    assert tie.sum() <= max(1, MAX_NEAR_TIE_FRAC * n_seq) or tie.mean() <= MAX_NEAR_TIE_FRAC, \
        f"{tie.sum()} near-tie sequences of {n_seq}"
    return int(tie.sum())


def gemm_err(y_gpu, y_ref):
    y = y_gpu.detach().float().cpu().double().numpy()
    rms = float(np.sqrt(np.mean(y_ref ** 2)))
    return float(np.abs(y - y_ref).max()) / rms
