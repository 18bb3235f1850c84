"""CPU oracle for the Uno draft+verify hot path -- TEST INFRASTRUCTURE ONLY.

Only tests/, the smoke check in __graft_entry__ and the CPU-baseline leg of
bench.py may import this package.  The product library never loads it and it
shares no code with the CUDA path: the arithmetic lives in uno_oracle.c (plain
fp64 loops, glibc exp/log, no fast-math, no FP contraction); this file only
compiles that C file with gcc and marshals numpy arrays into it.

Functions (each documented in uno_oracle.c with the passage it follows):
  gated_lora_linear(x, W, A, B, gate, alpha)  -> y (float64)
  verify_block(p_logits, q_logits, draft, u_accept, u_resample)  -> VerifyResult
  verify_block_ex(..., temperature, mode)  -> VerifyResult (temperature, inverse-CDF resample)
  lm_head_verify(h_p, h_q, W_p, W_q, draft, u_accept, u_resample)  -> VerifyResult (logits = h.W^T)
  tree_verify(logits, parent, token, u_accept, u_resample)  -> TreeResult (tree sampler)
  draft_sample(logits, u)  -> (tokens, status, margin)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "uno_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

GCC_FLAGS = ["-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
             "-shared", "-fPIC", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Compile uno_oracle.c into liboracle.so next to it (gcc)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *GCC_FLAGS, "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    lib.oracle_gated_lora_linear_f64.argtypes = [P, P, P, P, P, I64, I64, I64, I64,
                                                  ctypes.c_double, P]
    lib.oracle_gated_lora_linear_f64.restype = ctypes.c_int
    lib.oracle_verify_block_f64.argtypes = [P, P, P, P, P, I64, I64, I64, I64,
                                            P, P, P, P, P, P]
    lib.oracle_verify_block_f64.restype = ctypes.c_int
    lib.oracle_verify_block_ex_f64.argtypes = [P, P, P, P, P, I64, I64, I64, I64,
                                               ctypes.c_double, ctypes.c_int, P, P, P, P, P, P]
    lib.oracle_verify_block_ex_f64.restype = ctypes.c_int
    lib.oracle_lm_head_verify_f64.argtypes = [P, P, P, P, I64, P, P, P, I64, I64, I64, I64,
                                              P, P, P, P, P, P]
    lib.oracle_lm_head_verify_f64.restype = ctypes.c_int
    lib.oracle_tree_verify_f64.argtypes = [P, P, P, P, P, I64, I64, I64, P, P, P, P, P, P, P]
    lib.oracle_tree_verify_f64.restype = ctypes.c_int
    lib.oracle_draft_sample_f64.argtypes = [P, P, I64, I64, P, P, P]
    lib.oracle_draft_sample_f64.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    _lib = lib
    return lib


def _np(a, dtype):
    """Contiguous numpy copy/view of a numpy array or CPU torch tensor."""
    if hasattr(a, "detach"):
        a = a.detach().cpu()
        if dtype == np.float64:
            a = a.double()
        a = a.numpy()
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def gated_lora_linear(x, W, A, B, gate, alpha: float) -> np.ndarray:
    """y = x.W^T + gate * (alpha/rank) * (x.A^T).B^T in fp64."""
    lib = _load()
    x, W = _np(x, np.float64), _np(W, np.float64)
    A, B = _np(A, np.float64), _np(B, np.float64)
    g = _np(gate, np.uint8)
    M, d_in = x.shape
    d_out, rank = W.shape[0], A.shape[0]
    assert W.shape == (d_out, d_in) and A.shape == (rank, d_in)
    assert B.shape == (d_out, rank) and g.shape == (M,)
    y = np.zeros((M, d_out), dtype=np.float64)
    rc = lib.oracle_gated_lora_linear_f64(_ptr(x), _ptr(W), _ptr(A), _ptr(B), _ptr(g),
                                          M, d_in, d_out, rank, float(alpha), _ptr(y))
    if rc != 0:
        raise RuntimeError(f"oracle_gated_lora_linear_f64 failed: {rc}")
    return y


@dataclass
class VerifyResult:
    n_accepted: np.ndarray     # [Bn] int32
    out_tokens: np.ndarray     # [Bn, K+1] int32
    n_emitted: np.ndarray      # [Bn] int32
    status: np.ndarray         # [Bn] int32
    accept_margin: np.ndarray  # [Bn, K] float64, +inf where not evaluated
    race_margin: np.ndarray    # [Bn] float64, +inf where no race ran

    def near_tie(self, tol: float = 1e-4) -> np.ndarray:
        """[Bn] bool: a decision that fixed this sequence's output had an fp64
        margin below `tol` (an accept test at or before the stop position, or
        the race)."""
        acc = (self.accept_margin < tol).any(axis=1) if self.accept_margin.size else \
            np.zeros(self.n_accepted.shape, dtype=bool)
        return acc | (self.race_margin < tol)


def verify_block(p_logits, q_logits, draft, u_accept, u_resample) -> VerifyResult:
    lib = _load()
    p = _np(p_logits, np.float32)
    q = _np(q_logits, np.float32)
    Bn, Kp, V = p.shape
    K = q.shape[1]
    d = _np(draft, np.int32).reshape(Bn, K)
    ua = _np(u_accept, np.float32).reshape(Bn, K)
    ur = _np(u_resample, np.float32).reshape(Bn, V)
    n_acc = np.zeros(Bn, np.int32)
    toks = np.full((Bn, K + 1), -1, np.int32)
    n_em = np.zeros(Bn, np.int32)
    st = np.zeros(Bn, np.int32)
    am = np.full((Bn, K), np.inf)
    rm = np.full(Bn, np.inf)
    rc = lib.oracle_verify_block_f64(_ptr(p), _ptr(q), _ptr(d), _ptr(ua), _ptr(ur),
                                     Bn, K, Kp, V, _ptr(n_acc), _ptr(toks), _ptr(n_em),
                                     _ptr(st), _ptr(am), _ptr(rm))
    if rc != 0:
        raise RuntimeError(f"oracle_verify_block_f64 failed: {rc}")
    return VerifyResult(n_acc, toks, n_em, st, am, rm)


RESAMPLE_MODES = {"race": 0, "inverse_cdf": 1}


def verify_block_ex(p_logits, q_logits, draft, u_accept, u_resample, temperature: float = 1.0,
                    resample: str = "race") -> VerifyResult:
    """The verifier at temperature T with the resample drawn by the exponential
    race (u_resample [Bn, V]) or by the inverse CDF (u_resample [Bn]).  In
    inverse-CDF mode race_margin holds that sampler's bucket-edge margin."""
    lib = _load()
    mode = RESAMPLE_MODES[resample]
    p = _np(p_logits, np.float32)
    q = _np(q_logits, np.float32)
    Bn, Kp, V = p.shape
    K = q.shape[1]
    d = _np(draft, np.int32).reshape(Bn, K)
    ua = _np(u_accept, np.float32).reshape(Bn, K)
    ur = _np(u_resample, np.float32).reshape(Bn, V) if mode == 0 else \
        _np(u_resample, np.float32).reshape(Bn)
    n_acc = np.zeros(Bn, np.int32)
    toks = np.full((Bn, K + 1), -1, np.int32)
    n_em = np.zeros(Bn, np.int32)
    st = np.zeros(Bn, np.int32)
    am = np.full((Bn, K), np.inf)
    rm = np.full(Bn, np.inf)
    rc = lib.oracle_verify_block_ex_f64(_ptr(p), _ptr(q), _ptr(d), _ptr(ua), _ptr(ur),
                                        Bn, K, Kp, V, float(temperature), mode, _ptr(n_acc),
                                        _ptr(toks), _ptr(n_em), _ptr(st), _ptr(am), _ptr(rm))
    if rc != 0:
        raise RuntimeError(f"oracle_verify_block_ex_f64 failed: {rc}")
    return VerifyResult(n_acc, toks, n_em, st, am, rm)


def lm_head_verify(h_p, h_q, W_p, W_q, draft, u_accept, u_resample) -> VerifyResult:
    """The verifier on logits h.W^T (AR rows h_p [Bn,Kp,d] with head W_p [V,d],
    draft rows h_q [Bn,K,d] with head W_q [V,d]), everything in fp64."""
    lib = _load()
    hp, hq = _np(h_p, np.float64), _np(h_q, np.float64)
    Wp, Wq = _np(W_p, np.float64), _np(W_q, np.float64)
    Bn, Kp, d = hp.shape
    K = hq.shape[1]
    V = Wp.shape[0]
    assert Wp.shape == (V, d) and Wq.shape == (V, d) and hq.shape[2] == d
    dr = _np(draft, np.int32).reshape(Bn, K)
    ua = _np(u_accept, np.float32).reshape(Bn, K)
    ur = _np(u_resample, np.float32).reshape(Bn, V)
    n_acc = np.zeros(Bn, np.int32)
    toks = np.full((Bn, K + 1), -1, np.int32)
    n_em = np.zeros(Bn, np.int32)
    st = np.zeros(Bn, np.int32)
    am = np.full((Bn, K), np.inf)
    rm = np.full(Bn, np.inf)
    rc = lib.oracle_lm_head_verify_f64(_ptr(hp), _ptr(hq), _ptr(Wp), _ptr(Wq), d, _ptr(dr), _ptr(ua),
                                       _ptr(ur), Bn, K, Kp, V, _ptr(n_acc), _ptr(toks), _ptr(n_em),
                                       _ptr(st), _ptr(am), _ptr(rm))
    if rc != 0:
        raise RuntimeError(f"oracle_lm_head_verify_f64 failed: {rc}")
    return VerifyResult(n_acc, toks, n_em, st, am, rm)


@dataclass
class TreeResult:
    n_accepted: np.ndarray     # [Bn] int32, accepted depth
    path: np.ndarray           # [Bn, N] int32 accepted node ids, -1 padded
    out_tokens: np.ndarray     # [Bn, N+1] int32, -1 padded
    n_emitted: np.ndarray      # [Bn] int32
    status: np.ndarray         # [Bn] int32
    accept_margin: np.ndarray  # [Bn, N+1] float64, +inf for nodes not tested
    race_margin: np.ndarray    # [Bn] float64


def tree_verify(logits, parent, token, u_accept, u_resample) -> TreeResult:
    """Tree sampler's verification: logits [Bn, N+1, V] per node (node 0 the
    prefix), parent/token [Bn, N+1], u_accept [Bn, N+1], u_resample [Bn, V]."""
    lib = _load()
    lg = _np(logits, np.float32)
    Bn, N1, V = lg.shape
    N = N1 - 1
    par = _np(parent, np.int32).reshape(Bn, N1)
    tok = _np(token, np.int32).reshape(Bn, N1)
    ua = _np(u_accept, np.float32).reshape(Bn, N1)
    ur = _np(u_resample, np.float32).reshape(Bn, V)
    n_acc = np.zeros(Bn, np.int32)
    pth = np.full((Bn, N), -1, np.int32)
    toks = np.full((Bn, N1), -1, np.int32)
    n_em = np.zeros(Bn, np.int32)
    st = np.zeros(Bn, np.int32)
    am = np.full((Bn, N1), np.inf)
    rm = np.full(Bn, np.inf)
    rc = lib.oracle_tree_verify_f64(_ptr(lg), _ptr(par), _ptr(tok), _ptr(ua), _ptr(ur), Bn, N, V,
                                    _ptr(n_acc), _ptr(pth), _ptr(toks), _ptr(n_em), _ptr(st),
                                    _ptr(am), _ptr(rm))
    if rc != 0:
        raise RuntimeError(f"oracle_tree_verify_f64 failed: {rc}")
    return TreeResult(n_acc, pth, toks, n_em, st, am, rm)


def draft_sample(logits, u):
    """tokens[r] = argmax_v softmax(logits[r])(v) / (-ln u[r,v]).  Returns
    (tokens int32 [R], status int32 [R], margin float64 [R])."""
    lib = _load()
    lg = _np(logits, np.float32)
    V = lg.shape[-1]
    lg = lg.reshape(-1, V)
    R = lg.shape[0]
    uu = _np(u, np.float32).reshape(R, V)
    toks = np.zeros(R, np.int32)
    st = np.zeros(R, np.int32)
    mg = np.full(R, np.inf)
    rc = lib.oracle_draft_sample_f64(_ptr(lg), _ptr(uu), R, V, _ptr(toks), _ptr(st), _ptr(mg))
    if rc != 0:
        raise RuntimeError(f"oracle_draft_sample_f64 failed: {rc}")
    return toks, st, mg
