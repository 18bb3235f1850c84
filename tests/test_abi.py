"""Host-side checks of the C ABI (no GPU): libuno.so loads, exports every
function include/uno.h declares, and rejects bad arguments before touching
the device."""
import ctypes
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def L():
    from lossless_draft_verify_gated_b300 import build
    build.build()
    from lossless_draft_verify_gated_b300 import binding
    return binding.lib()


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(uno_\w+)\s*\(", src))
    return names


def test_every_declared_symbol_is_exported(L):
    from lossless_draft_verify_gated_b300 import binding
    declared = _declared_functions()
    assert {"uno_gated_lora_linear", "uno_verify_block", "uno_draft_sample"} <= declared
    for name in declared:
        assert hasattr(L, name), name
    # and the binding knows the signature of each
    assert declared == set(binding.SIGNATURES), declared ^ set(binding.SIGNATURES)


def test_status_strings(L):
    from lossless_draft_verify_gated_b300 import binding
    for code in range(0, -6, -1):
        s = binding.status_string(code)
        assert s and s != "unknown status"
    assert binding.status_string(-99) == "unknown status"
    assert binding.uno_version() >= 100


def test_workspace_queries_are_host_only(L):
    from lossless_draft_verify_gated_b300 import binding
    ws = binding.uno_gated_lora_linear_workspace(32, 4096, 4096, 128, binding.UNO_BF16)
    assert ws >= 32 * 128 * 2 and ws % 256 == 0
    assert binding.uno_gated_lora_linear_workspace(32, 4095, 4096, 128, binding.UNO_BF16) == 0
    assert binding.uno_gated_lora_linear_workspace(32, 4096, 4096, 512, binding.UNO_BF16) == 0
    v = binding.uno_verify_block_workspace(256, 16, 16, 128256)
    assert v > 0 and v % 256 == 0
    assert binding.uno_verify_block_workspace(2, 4, 6, 100) == 0  # Kp not in {K, K+1}
    assert binding.uno_verify_block_workspace(2, 0, 0, 100) == 0  # nothing to verify


def _lora(L, **kw):
    a = dict(x=16, W=16, A=16, B=16, gate=16, M=4, d_in=64, d_out=64, rank=16, alpha=32.0,
             dtype=1, y=16, ws=256, ws_bytes=1 << 20, stream=None)
    a.update(kw)
    P = lambda v: ctypes.c_void_p(v) if v else None  # noqa: E731
    return L.uno_gated_lora_linear(P(a["x"]), P(a["W"]), P(a["A"]), P(a["B"]), P(a["gate"]),
                                   a["M"], a["d_in"], a["d_out"], a["rank"], a["alpha"],
                                   a["dtype"], P(a["y"]), P(a["ws"]), a["ws_bytes"], a["stream"])


def test_lora_argument_errors(L):
    # every one of these is rejected on the host; none reaches a kernel
    assert _lora(L, x=0) == -1
    assert _lora(L, gate=0) == -1
    assert _lora(L, d_in=60) == -1
    assert _lora(L, rank=300) == -1
    assert _lora(L, d_out=0) == -1
    assert _lora(L, M=-1) == -1
    assert _lora(L, alpha=float("nan")) == -1
    assert _lora(L, dtype=7) == -3
    assert _lora(L, x=24) == -2
    assert _lora(L, ws=272) == -4
    assert _lora(L, ws_bytes=16) == -4
    assert _lora(L, M=0) == 0  # empty is a no-op


def test_verify_argument_errors(L):
    P = ctypes.c_void_p
    ptrs = [P(256)] * 5
    outs = [P(256)] * 4

    def call(Bn=2, K=4, Kp=4, V=100, ws=P(256), ws_bytes=1 << 20, p0=None):
        pp = list(ptrs)
        if p0 is not None:
            pp[0] = p0
        return L.uno_verify_block(*pp, Bn, K, Kp, V, *outs, ws, ws_bytes, None)

    assert call(Kp=6) == -1
    assert call(V=0) == -1
    assert call(K=300, Kp=300) == -1
    assert call(p0=P(0)) == -1
    assert call(p0=P(258)) == -2
    assert call(ws=P(264)) == -4
    assert call(ws_bytes=8) == -4
    assert call(Bn=0) == 0
    assert L.uno_draft_sample(None, None, 4, 10, None, None, None) == -1
    assert L.uno_draft_sample(None, None, 0, 10, None, None, None) == 0


def test_verify_ex_argument_errors(L):
    """uno_verify_block_ex: the temperature and the resample mode are checked on
    the host before anything else, then the same checks as uno_verify_block."""
    P = ctypes.c_void_p
    ptrs = [P(256)] * 5
    outs = [P(256)] * 4

    def call(T=1.0, mode=0, Bn=2, K=4, Kp=4, V=100, ws=P(256), ws_bytes=1 << 20, p0=None):
        pp = list(ptrs)
        if p0 is not None:
            pp[0] = p0
        return L.uno_verify_block_ex(*pp, Bn, K, Kp, V, T, mode, *outs, ws, ws_bytes, None)

    for T in (0.0, -1.0, float("inf"), float("nan")):
        assert call(T=T) == -1
    assert call(mode=2) == -1 and call(mode=-1) == -1
    assert call(T=0.5, Kp=6) == -1
    assert call(T=0.5, mode=1, p0=P(258)) == -2
    assert call(T=2.0, mode=1, ws=P(264)) == -4
    assert call(T=2.0, mode=1, ws_bytes=8) == -4
    assert call(T=0.7, mode=1, Bn=0) == 0


def test_batched_argument_errors(L):
    from lossless_draft_verify_gated_b300 import binding
    P = binding.LoraProblemC

    def arr(*ps):
        a = (P * len(ps))(*ps)
        return ctypes.cast(a, ctypes.c_void_p), a

    good = P(256, 256, 256, 256, 256, 256, 64, 64, 16, 32.0)
    a, keep = arr(good, good)
    ws = ctypes.c_void_p(256)
    assert L.uno_gated_lora_linear_batched(0, a, 4, 1, ws, 1 << 20, None) == -1
    assert L.uno_gated_lora_linear_batched(9, a, 4, 1, ws, 1 << 20, None) == -1
    bad = P(256, 256, 256, 256, 256, 256, 60, 64, 16, 32.0)  # d_in not a multiple of 8
    a2, keep2 = arr(good, bad)
    assert L.uno_gated_lora_linear_batched(2, a2, 4, 1, ws, 1 << 20, None) == -1
    mis = P(264, 256, 256, 256, 256, 256, 64, 64, 16, 32.0)
    a3, keep3 = arr(mis)
    assert L.uno_gated_lora_linear_batched(1, a3, 4, 1, ws, 1 << 20, None) == -2
    assert L.uno_gated_lora_linear_batched(2, a, 4, 1, ws, 16, None) == -4
    assert L.uno_gated_lora_linear_batched(2, a, 0, 1, ws, 16, None) == 0
    w1 = binding.uno_gated_lora_linear_batched_workspace([(4096, 4096, 128)] * 7, 32, 1)
    w2 = binding.uno_gated_lora_linear_workspace(32, 4096, 4096, 128, 1)
    assert w1 > w2 > 0


def test_tree_argument_errors(L):
    """uno_tree_verify: sizes, nulls, alignment and workspace checked on the host."""
    from lossless_draft_verify_gated_b300 import binding
    P = ctypes.c_void_p
    ins = [P(256)] * 5
    outs = [P(256)] * 5

    def call(Bn=2, N=4, V=100, ws=P(256), ws_bytes=1 << 20, l0=None, path=P(256)):
        ii = list(ins)
        if l0 is not None:
            ii[0] = l0
        oo = list(outs)
        oo[1] = path
        return L.uno_tree_verify(*ii, Bn, N, V, *oo, ws, ws_bytes, None)

    assert call(N=256) == -1 and call(N=-1) == -1 and call(V=0) == -1
    assert call(l0=P(0)) == -1
    assert call(path=None) == -1
    assert call(l0=P(258)) == -2
    assert call(ws=P(264)) == -4
    assert call(ws_bytes=8) == -4
    assert call(Bn=0) == 0
    w = binding.uno_tree_verify_workspace(4, 30, 128256)
    assert w > 0 and w % 256 == 0
    assert binding.uno_tree_verify_workspace(4, 256, 128256) == 0


def test_lm_head_argument_errors(L):
    """uno_lm_head_verify: mode, sizes (d and V multiples of 8), nulls,
    16-byte alignment of h, W and u_resample, workspace."""
    from lossless_draft_verify_gated_b300 import binding
    P = ctypes.c_void_p
    outs = [P(256)] * 4

    def call(Bn=2, K=4, Kp=4, V=1000, d=256, mode=0, h=P(256), W=P(256), ws=P(256),
             ws_bytes=1 << 30):
        return L.uno_lm_head_verify(h, W, P(256), P(256), P(256), Bn, K, Kp, V, d, mode, *outs, ws,
                                    ws_bytes, None)

    assert call(mode=4) == -1 and call(mode=-1) == -1
    assert call(V=1001) == -1 and call(d=100) == -1 and call(Kp=6) == -1
    assert call(h=None) == -1
    assert call(h=P(264)) == -2 and call(W=P(8)) == -2
    assert call(ws=P(264)) == -4 and call(ws_bytes=16) == -4
    assert call(Bn=0) == 0
    for mode in ("auto", "plain", "stats_store", "stats_recompute"):
        w = binding.uno_lm_head_verify_workspace(256, 16, 16, 128256, 4096, mode)
        assert w > 0 and w % 256 == 0
    # storing the logits takes 4 bytes per logit; recomputing the resampled rows does not
    big = binding.uno_lm_head_verify_workspace(256, 16, 16, 128256, 4096, "stats_store")
    small = binding.uno_lm_head_verify_workspace(256, 16, 16, 128256, 4096, "stats_recompute")
    assert big > 256 * 32 * 128256 * 4 > small
