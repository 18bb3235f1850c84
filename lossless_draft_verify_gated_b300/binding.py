"""ctypes binding of libuno.so with the same names as the C ABI (include/uno.h).

Argument marshalling only: tensors become device pointers, missing outputs and
workspaces are allocated with torch, the current torch stream is passed
through.  Every step of the computation runs in libuno.so's kernels; there is
no fallback.  If the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libuno.so")

UNO_OK = 0
UNO_ERR_ARG = -1
UNO_ERR_ALIGN = -2
UNO_ERR_UNSUPPORTED = -3
UNO_ERR_WORKSPACE = -4
UNO_ERR_CUDA = -5
UNO_F32 = 0
UNO_BF16 = 1
UNO_SEQ_OK = 0
UNO_SEQ_BAD_DRAFT = 1
UNO_SEQ_NONFINITE = 2

# Every function the header declares, with (restype, argtypes).
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int
_SZ = ctypes.c_size_t
SIGNATURES = {
    "uno_gated_lora_linear_workspace": (_SZ, [_I64, _I64, _I64, _I64, _I]),
    "uno_gated_lora_linear": (_I, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, ctypes.c_float, _I,
                                   _P, _P, _SZ, _P]),
    "uno_verify_block_workspace": (_SZ, [_I64, _I64, _I64, _I64]),
    "uno_verify_block": (_I, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _P, _P, _P, _P, _P, _SZ,
                              _P]),
    "uno_draft_sample": (_I, [_P, _P, _I64, _I64, _P, _P, _P]),
    "uno_verify_block_ex": (_I, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, ctypes.c_float, _I,
                                 _P, _P, _P, _P, _P, _SZ, _P]),
    "uno_verify_block_no_alloc_max_scratch": (_SZ, []),
    "uno_verify_block_no_alloc": (_I, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _P, _P, _P, _P,
                                       _P]),
    "uno_lm_head_verify_workspace": (_SZ, [_I64, _I64, _I64, _I64, _I64, _I]),
    "uno_lm_head_verify": (_I, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I, _P, _P, _P, _P,
                                _P, _SZ, _P]),
    "uno_tree_verify_workspace": (_SZ, [_I64, _I64, _I64]),
    "uno_tree_verify": (_I, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "uno_device_error": (_I, [_I]),
    "uno_status_string": (ctypes.c_char_p, [_I]),
    "uno_version": (_I, []),
}



class LoraProblemC(ctypes.Structure):
    """uno_lora_problem (include/uno.h)."""
    _fields_ = [("x", _P), ("W", _P), ("A", _P), ("B", _P), ("gate", _P), ("y", _P),
                ("d_in", _I64), ("d_out", _I64), ("rank", _I64), ("alpha", ctypes.c_float)]


SIGNATURES["uno_gated_lora_linear_batched_workspace"] = (_SZ, [_I, _P, _I64, _I])
SIGNATURES["uno_gated_lora_linear_batched"] = (_I, [_I, _P, _I64, _I, _P, _SZ, _P])
SIGNATURES["uno_lora_plan_check"] = (_I, [_I, _P, _I64, _I, _I])


def uno_lora_plan_check(shapes, M: int, sms: int, dtype: int = 1) -> int:
    """Host-only check of the projection schedule for problems given as
    (d_in, d_out, rank) on a GPU with `sms` SMs: 0 when its invariants hold."""
    arr = (LoraProblemC * len(shapes))()
    for i, (di, do, r) in enumerate(shapes):
        arr[i] = LoraProblemC(0, 0, 0, 0, 0, 0, di, do, r, 1.0)
    return int(lib().uno_lora_plan_check(len(shapes), ctypes.cast(arr, _P), M, dtype, sms))

_lib = None


class UnoError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} failed: {code} ({status_string(code)})")
        self.code = code


def lib() -> ctypes.CDLL:
    """Load libuno.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libuno.so not built ({LIB_PATH}); run "
                               "`python -m lossless_draft_verify_gated_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().uno_status_string(int(code)).decode()


def _dptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libuno takes CUDA tensors only")
    if not t.is_contiguous():
        raise ValueError("libuno takes contiguous tensors only")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(fn, rc):
    if rc != UNO_OK:
        raise UnoError(fn, rc)


def _workspace(nbytes: int, device) -> torch.Tensor:
    # torch's caching allocator returns 512-byte aligned blocks
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


_DT = {torch.float32: UNO_F32, torch.bfloat16: UNO_BF16}


def uno_gated_lora_linear_workspace(M, d_in, d_out, rank, dtype) -> int:
    dt = _DT[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return int(lib().uno_gated_lora_linear_workspace(M, d_in, d_out, rank, dt))


def uno_gated_lora_linear(x, W, A, B, gate, alpha, *, y=None, workspace=None, stream=None):
    """y = x.W^T + gate * (alpha/rank) * (x.A^T).B^T (see include/uno.h)."""
    M, d_in = x.shape
    d_out = W.shape[0]
    rank = A.shape[0]
    dt = _DT[x.dtype]
    if y is None:
        y = torch.empty((M, d_out), dtype=x.dtype, device=x.device)
    if workspace is None:
        workspace = _workspace(uno_gated_lora_linear_workspace(M, d_in, d_out, rank, dt), x.device)
    rc = lib().uno_gated_lora_linear(_dptr(x), _dptr(W), _dptr(A), _dptr(B), _dptr(gate), M, d_in,
                                     d_out, rank, float(alpha), dt, _dptr(y), _dptr(workspace),
                                     workspace.numel(), _stream(stream))
    _check("uno_gated_lora_linear", rc)
    return y


_PROBLEM_ARRAYS = {}


def _problems(problems):
    # repeated calls with the same tensors (a decode loop) reuse the marshalled array
    key = tuple((t.data_ptr(), tuple(t.shape), t.device.index, t.is_contiguous()) for p in problems
                for t in (p[0], p[1], p[2], p[3], p[4], p[6])) + tuple(float(p[5]) for p in problems)
    arr = _PROBLEM_ARRAYS.get(key)
    if arr is not None:
        return arr
    arr = _marshal_problems(problems)
    if len(_PROBLEM_ARRAYS) > 64:
        _PROBLEM_ARRAYS.clear()
    _PROBLEM_ARRAYS[key] = arr
    return arr


def _marshal_problems(problems):
    arr = (LoraProblemC * len(problems))()
    for i, (x, W, A, B, gate, alpha, y) in enumerate(problems):
        for t in (x, W, gate, y) + ((A, B) if A.numel() else ()):
            _dptr(t)  # device and contiguity checks
        arr[i] = LoraProblemC(x.data_ptr(), W.data_ptr(), A.data_ptr() if A.numel() else 0,
                              B.data_ptr() if B.numel() else 0, gate.data_ptr(), y.data_ptr(),
                              x.shape[1], W.shape[0], A.shape[0], float(alpha))
    return arr


def uno_gated_lora_linear_batched_workspace(shapes, M, dtype) -> int:
    """shapes: list of (d_in, d_out, rank)."""
    dt = _DT[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    arr = (LoraProblemC * len(shapes))()
    for i, (di, do, r) in enumerate(shapes):
        arr[i] = LoraProblemC(0, 0, 0, 0, 0, 0, di, do, r, 1.0)
    return int(lib().uno_gated_lora_linear_batched_workspace(len(shapes), ctypes.cast(arr, _P), M, dt))


def uno_gated_lora_linear_batched(problems, *, workspace=None, stream=None):
    """problems: list of (x, W, A, B, gate, alpha, y) tensors, all with the same
    row count M and dtype.  One persistent kernel computes every y in place."""
    x0 = problems[0][0]
    M = x0.shape[0]
    dt = _DT[x0.dtype]
    arr = _problems(problems)
    if workspace is None:
        shapes = [(p[0].shape[1], p[1].shape[0], p[2].shape[0]) for p in problems]
        workspace = _workspace(uno_gated_lora_linear_batched_workspace(shapes, M, dt), x0.device)
    rc = lib().uno_gated_lora_linear_batched(len(problems), ctypes.cast(arr, _P), M, dt,
                                             _dptr(workspace), workspace.numel(), _stream(stream))
    _check("uno_gated_lora_linear_batched", rc)
    return [p[6] for p in problems]


def uno_verify_block_workspace(Bn, K, Kp, V) -> int:
    return int(lib().uno_verify_block_workspace(Bn, K, Kp, V))


def uno_verify_block(p_logits, q_logits, draft, u_accept, u_resample, *, out=None, workspace=None,
                     stream=None):
    """Returns (n_accepted [Bn], out_tokens [Bn, K+1], n_emitted [Bn], status [Bn]), int32."""
    Bn, Kp, V = p_logits.shape
    K = q_logits.shape[1]
    dev = p_logits.device
    if out is None:
        out = (torch.empty(Bn, dtype=torch.int32, device=dev),
               torch.empty((Bn, K + 1), dtype=torch.int32, device=dev),
               torch.empty(Bn, dtype=torch.int32, device=dev),
               torch.empty(Bn, dtype=torch.int32, device=dev))
    n_acc, toks, n_em, st = out
    if workspace is None:
        workspace = _workspace(uno_verify_block_workspace(Bn, K, Kp, V), dev)
    rc = lib().uno_verify_block(_dptr(p_logits), _dptr(q_logits), _dptr(draft), _dptr(u_accept),
                                _dptr(u_resample), Bn, K, Kp, V, _dptr(n_acc), _dptr(toks),
                                _dptr(n_em), _dptr(st), _dptr(workspace), workspace.numel(),
                                _stream(stream))
    _check("uno_verify_block", rc)
    return n_acc, toks, n_em, st


UNO_RESAMPLE_RACE = 0
UNO_RESAMPLE_INVERSE_CDF = 1
_RESAMPLE = {"race": UNO_RESAMPLE_RACE, "inverse_cdf": UNO_RESAMPLE_INVERSE_CDF}


def uno_verify_block_ex(p_logits, q_logits, draft, u_accept, u_resample, *, temperature=1.0,
                        resample="race", out=None, workspace=None, stream=None):
    """The verifier at `temperature`, resampling by "race" (u_resample [Bn, V])
    or "inverse_cdf" (u_resample [Bn]).  Returns (n_accepted, out_tokens,
    n_emitted, status), int32."""
    Bn, Kp, V = p_logits.shape
    K = q_logits.shape[1]
    dev = p_logits.device
    if out is None:
        out = (torch.empty(Bn, dtype=torch.int32, device=dev),
               torch.empty((Bn, K + 1), dtype=torch.int32, device=dev),
               torch.empty(Bn, dtype=torch.int32, device=dev),
               torch.empty(Bn, dtype=torch.int32, device=dev))
    n_acc, toks, n_em, st = out
    if workspace is None:
        workspace = _workspace(uno_verify_block_workspace(Bn, K, Kp, V), dev)
    rc = lib().uno_verify_block_ex(_dptr(p_logits), _dptr(q_logits), _dptr(draft), _dptr(u_accept),
                                   _dptr(u_resample), Bn, K, Kp, V, float(temperature),
                                   _RESAMPLE[resample], _dptr(n_acc), _dptr(toks), _dptr(n_em),
                                   _dptr(st), _dptr(workspace), workspace.numel(), _stream(stream))
    _check("uno_verify_block_ex", rc)
    return n_acc, toks, n_em, st


UNO_LM_AUTO = 0
UNO_LM_PLAIN = 1
UNO_LM_STATS_STORE = 2
UNO_LM_STATS_RECOMPUTE = 3
_LM_MODE = {"auto": UNO_LM_AUTO, "plain": UNO_LM_PLAIN, "stats_store": UNO_LM_STATS_STORE,
            "stats_recompute": UNO_LM_STATS_RECOMPUTE}


def uno_lm_head_verify_workspace(Bn, K, Kp, V, d, mode="auto") -> int:
    return int(lib().uno_lm_head_verify_workspace(Bn, K, Kp, V, d, _LM_MODE[mode]))


def uno_lm_head_verify(h, W, draft, u_accept, u_resample, *, Kp=None, mode="auto", out=None,
                       workspace=None, stream=None):
    """LM head + block verifier.  h [Bn*Kp + Bn*K, d] bf16 (AR rows of every
    sequence, then draft rows), W [V, d] bf16, draft/u_accept [Bn, K],
    u_resample [Bn, V].  Returns (n_accepted, out_tokens, n_emitted, status)."""
    Bn, K = draft.shape
    Kp = K if Kp is None else Kp
    V, d = W.shape
    assert h.shape == (Bn * (Kp + K), d)
    dev = h.device
    if out is None:
        out = (torch.empty(Bn, dtype=torch.int32, device=dev),
               torch.empty((Bn, K + 1), dtype=torch.int32, device=dev),
               torch.empty(Bn, dtype=torch.int32, device=dev),
               torch.empty(Bn, dtype=torch.int32, device=dev))
    n_acc, toks, n_em, st = out
    if workspace is None:
        workspace = _workspace(uno_lm_head_verify_workspace(Bn, K, Kp, V, d, mode), dev)
    rc = lib().uno_lm_head_verify(_dptr(h), _dptr(W), _dptr(draft), _dptr(u_accept),
                                  _dptr(u_resample), Bn, K, Kp, V, d, _LM_MODE[mode], _dptr(n_acc),
                                  _dptr(toks), _dptr(n_em), _dptr(st), _dptr(workspace),
                                  workspace.numel(), _stream(stream))
    _check("uno_lm_head_verify", rc)
    return n_acc, toks, n_em, st


def uno_tree_verify_workspace(Bn, N, V) -> int:
    return int(lib().uno_tree_verify_workspace(Bn, N, V))


def uno_tree_verify(logits, parent, token, u_accept, u_resample, *, out=None, workspace=None,
                    stream=None):
    """Tree sampler's verification.  logits [Bn, N+1, V], parent/token/u_accept
    [Bn, N+1], u_resample [Bn, V].  Returns (n_accepted [Bn], path [Bn, N],
    out_tokens [Bn, N+1], n_emitted [Bn], status [Bn]), int32."""
    Bn, N1, V = logits.shape
    N = N1 - 1
    dev = logits.device
    if out is None:
        out = (torch.empty(Bn, dtype=torch.int32, device=dev),
               torch.empty((Bn, N), dtype=torch.int32, device=dev),
               torch.empty((Bn, N1), dtype=torch.int32, device=dev),
               torch.empty(Bn, dtype=torch.int32, device=dev),
               torch.empty(Bn, dtype=torch.int32, device=dev))
    n_acc, pth, toks, n_em, st = out
    if workspace is None:
        workspace = _workspace(uno_tree_verify_workspace(Bn, N, V), dev)
    rc = lib().uno_tree_verify(_dptr(logits), _dptr(parent), _dptr(token), _dptr(u_accept),
                               _dptr(u_resample), Bn, N, V, _dptr(n_acc),
                               _dptr(pth) if N > 0 else None, _dptr(toks), _dptr(n_em), _dptr(st),
                               _dptr(workspace), workspace.numel(), _stream(stream))
    _check("uno_tree_verify", rc)
    return n_acc, pth, toks, n_em, st


def uno_draft_sample(logits, u, *, tokens=None, status=None, stream=None):
    """tokens[r] ~ softmax(logits[r]) via the exponential race on u.  Returns (tokens, status)."""
    V = logits.shape[-1]
    R = logits.numel() // V if V else 0
    shape = logits.shape[:-1]
    if tokens is None:
        tokens = torch.empty(shape, dtype=torch.int32, device=logits.device)
    if status is None:
        status = torch.empty(shape, dtype=torch.int32, device=logits.device)
    rc = lib().uno_draft_sample(_dptr(logits), _dptr(u), R, V, _dptr(tokens), _dptr(status),
                                _stream(stream))
    _check("uno_draft_sample", rc)
    return tokens, status


def uno_device_error(reset: bool = False) -> int:
    return int(lib().uno_device_error(1 if reset else 0))


def uno_version() -> int:
    return int(lib().uno_version())
