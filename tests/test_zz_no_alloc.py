"""The block verifier entry point that allocates nothing.

Callers that cannot allocate device memory (an op inside another runtime that
gets only its input and output buffers, a serving path whose memory pool it may
not grow) call uno_verify_block_no_alloc, which keeps its scratch in a fixed
array inside libuno.so.  This test calls it through the C ABI, twice in a row
on different inputs (the array keeps the previous call's contents), and checks
that its outputs equal those of uno_verify_block, which takes a caller
workspace.  The outputs are integers, so the comparison is exact.

Collected last on purpose (file name), so that a failure here leaves every
other test already run."""
import ctypes

import pytest
import torch

from lossless_draft_verify_gated_b300 import inputs

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _no_alloc(L, p, q, d, ua, ur):
    Bn, Kp, V = p.shape
    K = q.shape[1]
    outs = [torch.full((Bn,), -9, dtype=torch.int32, device="cuda"),
            torch.full((Bn, K + 1), -9, dtype=torch.int32, device="cuda"),
            torch.full((Bn,), -9, dtype=torch.int32, device="cuda"),
            torch.full((Bn,), -9, dtype=torch.int32, device="cuda")]
    rc = L.uno_verify_block_no_alloc(_ptr(p), _ptr(q), _ptr(d), _ptr(ua), _ptr(ur), Bn, K, Kp, V,
                                     *[_ptr(o) for o in outs],
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, rc
    return outs


def test_no_alloc_matches_workspace_entry_point():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lossless_draft_verify_gated_b300 import binding, build
    build.build()
    L = binding.lib()
    assert L.uno_verify_block_no_alloc_max_scratch() == 8 << 20
    cases = [(64, 16, 128256, None, 1.0, 11), (7, 5, 4099, 6, 4.0, 12)]  # two calls in a row
    for Bn, K, V, Kp, sigma, seed in cases:
        pr = inputs.verify_problem(Bn, K, V, Kp=Kp, sigma=sigma, seed=seed, device="cuda")
        draft, st = binding.uno_draft_sample(pr.q_logits, pr.u_draft)
        assert int(st.abs().sum()) == 0
        args = (pr.p_logits, pr.q_logits, draft, pr.u_accept, pr.u_resample)
        ref = binding.uno_verify_block(*args)
        got = _no_alloc(L, *args)
        torch.cuda.synchronize()
        for a, b in zip(ref, got):
            assert torch.equal(a, b)
    # sizes beyond the array are refused up front, with nothing launched
    big_B = 1 << 24
    need = binding.uno_verify_block_workspace(big_B, 16, 16, 128256)
    assert need > 8 << 20
    one = torch.zeros(1, device="cuda")
    oi = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = L.uno_verify_block_no_alloc(_ptr(one), _ptr(one), _ptr(oi), _ptr(one), _ptr(one), big_B, 16,
                                     16, 128256, _ptr(oi), _ptr(oi), _ptr(oi), _ptr(oi), None)
    assert rc == binding.UNO_ERR_WORKSPACE
