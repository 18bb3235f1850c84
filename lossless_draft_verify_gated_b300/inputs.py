"""Seeded synthetic inputs for the gated-LoRA projection and the block verifier.

This module only draws random numbers with the shapes and distributions of the
workloads; it holds none of the method's arithmetic.  Both the CUDA path and
the CPU oracle are fed from here, so that the two sides read identical bits.

Distributions (a Llama-3-8B-shaped layer with a rank-128, alpha=256 adapter,
the size "Unlocking Lossless Speedups in LLMs via Discrete Diffusion"
(aifromscratch.in), section "Two Decoupled Weight Sets", gives for the
diffusion weights):
  x ~ N(0,1), W ~ N(0, 0.02), A ~ N(0, 0.02), B ~ N(0, b_std)
  AR logits ~ N(0, 3); draft logits = AR logits + N(0, sigma)
Uniforms are multiples of 2^-24 so that every value is exact in fp32:
  u_accept in [0, 1)      : k * 2^-24, k in [0, 2^24)
  u_race   in (0, 1)      : k * 2^-24, k in [1, 2^24)   (never 0, never 1)
"""
from __future__ import annotations

import zlib
from dataclasses import dataclass

import torch

BASE_SEED = 1234
_TWO24 = 1 << 24

# Llama-3-8B-shaped projections (d_in, d_out), in layer order.
LLAMA3_8B_PROJECTIONS = (
    ("q", 4096, 4096),
    ("k", 4096, 1024),
    ("v", 4096, 1024),
    ("o", 4096, 4096),
    ("gate", 4096, 14336),
    ("up", 4096, 14336),
    ("down", 14336, 4096),
)
# Which synthetic activation feeds which projection (attention/MLP are not on
# the path, so each block of projections gets its own seeded input).
LLAMA3_8B_INPUT_OF = {"q": "attn_in", "k": "attn_in", "v": "attn_in",
                      "o": "o_in", "gate": "mlp_in", "up": "mlp_in",
                      "down": "down_in"}


def generator(name: str, seed: int = BASE_SEED, device: str | torch.device = "cpu") -> torch.Generator:
    """A torch.Generator seeded from (seed, name) by a stable hash."""
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + zlib.crc32(name.encode())) & 0x7FFF_FFFF_FFFF)
    return g


def gate_mask(M: int, block: int, device="cpu") -> torch.Tensor:
    """uint8 gate per row: rows alternate in runs of `block`, verification
    rows (0) first, then draft rows (1), e.g. block=16, M=32: 16 zeros, 16 ones."""
    m = torch.arange(M, device=device)
    return ((m // block) % 2).to(torch.uint8)


def normal(shape, std: float, name: str, seed: int = BASE_SEED, dtype=torch.float32,
           device="cpu") -> torch.Tensor:
    g = generator(name, seed, device)
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def uniform_accept(shape, name: str, seed: int = BASE_SEED, device="cpu") -> torch.Tensor:
    """float32 in [0,1): k * 2^-24 with k uniform in [0, 2^24)."""
    g = generator(name, seed, device)
    k = torch.randint(0, _TWO24, tuple(shape), generator=g, device=device, dtype=torch.int32)
    return k.to(torch.float32).mul_(1.0 / _TWO24)


def uniform_race(shape, name: str, seed: int = BASE_SEED, device="cpu") -> torch.Tensor:
    """float32 in (0,1): k * 2^-24 with k uniform in [1, 2^24)."""
    g = generator(name, seed, device)
    k = torch.randint(1, _TWO24, tuple(shape), generator=g, device=device, dtype=torch.int32)
    return k.to(torch.float32).mul_(1.0 / _TWO24)


@dataclass
class LoraProblem:
    x: torch.Tensor
    W: torch.Tensor
    A: torch.Tensor
    B: torch.Tensor
    gate: torch.Tensor
    alpha: float

    @property
    def shape(self):
        M, d_in = self.x.shape
        return M, d_in, self.W.shape[0], self.A.shape[0]


def lora_problem(M: int, d_in: int, d_out: int, rank: int, alpha: float, *,
                 dtype=torch.bfloat16, block: int = 16, seed: int = BASE_SEED,
                 name: str = "proj", b_std: float = 0.02, w_std: float = 0.02,
                 a_std: float = 0.02, x_name: str | None = None,
                 device="cpu") -> LoraProblem:
    """One gated-LoRA projection's inputs.  `x_name` lets several projections
    share one activation (q/k/v read the same layer input)."""
    xn = x_name or f"{name}.x"
    x = normal((M, d_in), 1.0, f"{xn}.M{M}.d{d_in}", seed, dtype, device)
    W = normal((d_out, d_in), w_std, f"{name}.W", seed, dtype, device)
    A = normal((rank, d_in), a_std, f"{name}.A", seed, dtype, device)
    B = normal((d_out, rank), b_std, f"{name}.B", seed, dtype, device)
    return LoraProblem(x, W, A, B, gate_mask(M, block, device), float(alpha))


def llama3_layer(M: int, *, rank: int = 128, alpha: float = 256.0, block: int = 16,
                 seed: int = BASE_SEED, dtype=torch.bfloat16, device="cpu"):
    """The 7 projections of one Llama-3-8B-shaped layer at M rows.  Projections
    that read the same layer input (q/k/v, gate/up) share one x tensor, and all
    share one gate tensor, as in the layer itself."""
    out, xs, gate = [], {}, None
    for n, di, do in LLAMA3_8B_PROJECTIONS:
        pr = lora_problem(M, di, do, rank, alpha, dtype=dtype, block=block, seed=seed,
                          name=f"llama3.{n}", x_name=f"llama3.{LLAMA3_8B_INPUT_OF[n]}", device=device)
        key = LLAMA3_8B_INPUT_OF[n]
        if key in xs:
            pr.x = xs[key]  # same seed and name: identical values, one tensor
        else:
            xs[key] = pr.x
        gate = pr.gate if gate is None else gate
        pr.gate = gate
        out.append((n, pr))
    return out


@dataclass
class VerifyProblem:
    p_logits: torch.Tensor   # [Bn, Kp, V] float32
    q_logits: torch.Tensor   # [Bn, K, V]  float32
    u_accept: torch.Tensor   # [Bn, K]     float32 in [0,1)
    u_resample: torch.Tensor  # [Bn, V]    float32 in (0,1)
    u_draft: torch.Tensor    # [Bn, K, V]  float32 in (0,1): drives draft sampling

    @property
    def shape(self):
        Bn, Kp, V = self.p_logits.shape
        return Bn, self.q_logits.shape[1], Kp, V


def verify_problem(Bn: int, K: int, V: int, *, Kp: int | None = None, sigma: float = 1.0,
                   p_std: float = 3.0, seed: int = BASE_SEED, device="cpu",
                   with_u_draft: bool = True) -> VerifyProblem:
    """AR logits ~ N(0, p_std); draft logits = AR logits (first K rows) + N(0, sigma)."""
    Kp = K if Kp is None else Kp
    tag = f"B{Bn}.K{K}.Kp{Kp}.V{V}.s{sigma}"
    p = normal((Bn, Kp, V), p_std, f"verify.p.{tag}", seed, torch.float32, device)
    q = p[:, :K].clone()
    q.add_(normal((Bn, K, V), sigma, f"verify.dq.{tag}", seed, torch.float32, device))
    ua = uniform_accept((Bn, K), f"verify.ua.{tag}", seed, device)
    ur = uniform_race((Bn, V), f"verify.ur.{tag}", seed, device)
    ud = (uniform_race((Bn, K, V), f"verify.ud.{tag}", seed, device) if with_u_draft
          else torch.empty(0, device=device))
    return VerifyProblem(p, q, ua, ur, ud)


@dataclass
class LmHeadProblem:
    h: torch.Tensor           # [Bn*Kp + Bn*K, d] bf16: AR rows of every sequence, then draft rows
    W: torch.Tensor           # [V, d] bf16 LM head
    u_accept: torch.Tensor    # [Bn, K]
    u_resample: torch.Tensor  # [Bn, V]
    u_draft: torch.Tensor     # [Bn, K, V]
    Bn: int
    K: int
    Kp: int


def lm_head_problem(Bn: int, K: int, V: int, d: int, *, Kp: int | None = None, sigma: float = 1.0,
                    logit_std: float = 3.0, seed: int = BASE_SEED, device="cpu") -> LmHeadProblem:
    """Final hidden states and an LM head whose logits have the verifier's
    workload statistics: AR hidden states ~ N(0, 1), W ~ N(0, logit_std/sqrt(d))
    (logits ~ N(0, logit_std)); the draft rows' hidden states are the AR rows'
    plus N(0, sigma/logit_std), so draft logits are AR logits plus about
    N(0, sigma)."""
    Kp = K if Kp is None else Kp
    tag = f"B{Bn}.K{K}.Kp{Kp}.V{V}.d{d}.s{sigma}"
    ha = normal((Bn, Kp, d), 1.0, f"lm.ha.{tag}", seed, torch.float32, device)
    hd = ha[:, :K] + normal((Bn, K, d), sigma / logit_std, f"lm.hd.{tag}", seed, torch.float32, device)
    h = torch.cat([ha.reshape(Bn * Kp, d), hd.reshape(Bn * K, d)]).to(torch.bfloat16)
    W = normal((V, d), logit_std / d ** 0.5, f"lm.W.V{V}.d{d}", seed, torch.bfloat16, device)
    ua = uniform_accept((Bn, K), f"lm.ua.{tag}", seed, device)
    ur = uniform_race((Bn, V), f"lm.ur.{tag}", seed, device)
    ud = uniform_race((Bn, K, V), f"lm.ud.{tag}", seed, device)
    return LmHeadProblem(h, W, ua, ur, ud, Bn, K, Kp)
