"""GPU parity of the gated-LoRA projection against the fp64 oracle:
max |y_gpu - y_ref| <= 2e-2 * rms(y_ref) with bf16 operands and fp32
accumulation, plus the exact structural properties of the gate.
("Unlocking Lossless Speedups in LLMs via Discrete Diffusion",
aifromscratch.in, section "Two Decoupled Weight Sets".)"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import GEMM_TOL, gemm_err, require_gpu
from lossless_draft_verify_gated_b300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _gpu_run(pr, **kw):
    from lossless_draft_verify_gated_b300 import uno_gated_lora_linear
    d = "cuda"
    y = uno_gated_lora_linear(pr.x.to(d), pr.W.to(d), pr.A.to(d), pr.B.to(d), pr.gate.to(d),
                              pr.alpha, **kw)
    torch.cuda.synchronize()
    return y


def _ref(pr, rows=None):
    x, g = (pr.x, pr.gate) if rows is None else (pr.x[rows], pr.gate[rows])
    return oracle.gated_lora_linear(x, pr.W, pr.A, pr.B, g, pr.alpha)


@pytest.mark.parametrize("M,d_in,d_out,r,alpha,dtype,block", [
    (16, 256, 256, 16, 32.0, torch.float32, 4),     # tiny smoke configuration (fp32 in/out)
    (16, 256, 256, 16, 32.0, torch.bfloat16, 4),
    (13, 200, 136, 24, 48.0, torch.bfloat16, 4),    # ragged M, K tail, N tail, rank not /64
    (32, 4096, 1024, 128, 256.0, torch.bfloat16, 16),  # k/v projection shape at decode M
    (100, 512, 384, 128, 256.0, torch.bfloat16, 16),   # swap path, 128-wide token tile
    (256, 1024, 520, 64, 128.0, torch.bfloat16, 16),   # large-M order, fewer tiles than CTAs
    (300, 512, 1000, 128, 256.0, torch.bfloat16, 16),  # non-swap path, ragged M and N
    (40, 64, 64, 8, 16.0, torch.bfloat16, 16),         # single K-block
    (48, 512, 256, 256, 512.0, torch.bfloat16, 16),    # rank 256: two 128-row passes of the split-K adapter
    (32, 16384, 64, 256, 512.0, torch.bfloat16, 16),   # split-K adapter chunks staged in several rounds
    (256, 14336, 1024, 128, 256.0, torch.bfloat16, 16),  # long T tiles, each in many pieces (token-rows order)
    (384, 1024, 512, 256, 512.0, torch.bfloat16, 16),    # rank 256 in token-rows order: 32 slices per T tile
    # pair order (256-token tiles by CTA pairs, M > 128 with little padding and
    # a tile for at least half of the pairs): ragged M and N, small ranks whose
    # T tiles split into 16- and 32-row halves, rank 256, fp32 operands
    (2660, 512, 1000, 64, 128.0, torch.bfloat16, 16),
    (8192, 256, 256, 32, 64.0, torch.bfloat16, 16),
    (4096, 768, 520, 256, 512.0, torch.bfloat16, 16),
    (4096, 512, 512, 128, 256.0, torch.float32, 16),
])
def test_lora_parity(M, d_in, d_out, r, alpha, dtype, block):
    pr = inputs.lora_problem(M, d_in, d_out, r, alpha, dtype=dtype, block=block,
                             name=f"t.{M}.{d_in}.{d_out}.{r}")
    y = _gpu_run(pr)
    assert y.dtype == dtype and y.shape == (M, d_out)
    ref = _ref(pr)
    assert gemm_err(y, ref) <= GEMM_TOL
    # the adapter term is really there: the error against the base GEMM alone is large
    base = oracle.gated_lora_linear(pr.x, pr.W, pr.A, pr.B, torch.zeros_like(pr.gate), pr.alpha)
    if pr.gate.any():
        assert gemm_err(y, base) > 5 * gemm_err(y, ref)


@pytest.mark.parametrize("name,d_in,d_out", inputs.LLAMA3_8B_PROJECTIONS)
def test_llama3_layer_decode_parity(name, d_in, d_out):
    """Each projection of the Llama-3-8B-shaped layer at batch 1 x block 16 (M = 32)."""
    pr = inputs.lora_problem(32, d_in, d_out, 128, 256.0, block=16, name=f"llama3.{name}",
                             x_name=f"llama3.{inputs.LLAMA3_8B_INPUT_OF[name]}")
    y = _gpu_run(pr)
    assert gemm_err(y, _ref(pr)) <= GEMM_TOL


@pytest.mark.parametrize("M", [2048])
@pytest.mark.parametrize("name,d_in,d_out", [inputs.LLAMA3_8B_PROJECTIONS[0],
                                             inputs.LLAMA3_8B_PROJECTIONS[4],
                                             inputs.LLAMA3_8B_PROJECTIONS[6]])
def test_llama3_layer_large_m_sampled(M, name, d_in, d_out):
    """Batch 64 x block 16 (M = 2048): 64 seeded rows (half gate 0, half gate 1)
    are checked against the oracle over every column."""
    pr = inputs.lora_problem(M, d_in, d_out, 128, 256.0, block=16, name=f"llama3.{name}",
                             x_name=f"llama3.{inputs.LLAMA3_8B_INPUT_OF[name]}")
    y = _gpu_run(pr)
    g = inputs.generator(f"rows.{name}.{M}")
    rows = torch.randperm(M, generator=g)[:64]
    ref = _ref(pr, rows)
    assert gemm_err(y[rows.cuda()], ref) <= GEMM_TOL
    assert pr.gate[rows].sum() > 0 and (pr.gate[rows] == 0).sum() > 0


@pytest.mark.parametrize("M", [64, 128, 129, 255])
def test_operand_order_boundaries(M):
    """Both sides of the decode/large-M switch (tokens as the MMA N side up to
    128 rows, as its M side above) and the per-piece adapter at N = 64 and
    N = 128: a q-shaped projection alone (per-piece T) and the gate/up pair
    (shared T), every row against the oracle."""
    pr = inputs.lora_problem(M, 4096, 4096, 128, 256.0, block=16, name=f"bnd.q.{M}")
    assert gemm_err(_gpu_run(pr), _ref(pr)) <= GEMM_TOL
    prs = [inputs.lora_problem(M, 4096, 14336, 128, 256.0, block=16, name=f"bnd.gu{i}.{M}")
           for i in range(2)]
    rows = torch.randperm(M, generator=inputs.generator(f"bnd.rows.{M}"))[:24]
    for pr, y in zip(prs, _batched(prs)):
        assert gemm_err(y[rows.cuda()], _ref(pr, rows)) <= GEMM_TOL


def test_large_m_deterministic_and_gate_zero_rows():
    """Data-parallel waves at M = 2048 (the pair order, 256-token tiles by CTA
    pairs): two calls give the same bits, and gate-0 rows equal a call with
    every gate 0."""
    pr = inputs.lora_problem(2048, 4096, 4096, 128, 256.0, block=16, name="det.large")
    a, b = _gpu_run(pr), _gpu_run(pr)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    pr0 = inputs.LoraProblem(pr.x, pr.W, pr.A, pr.B, torch.zeros_like(pr.gate), pr.alpha)
    z = (pr.gate == 0).cuda()
    assert torch.equal(a[z].view(torch.int16), _gpu_run(pr0)[z].view(torch.int16))


def test_gate_zero_rows_bit_equal_all_gates_zero():
    pr = inputs.lora_problem(32, 4096, 4096, 128, 256.0, name="gz")
    y = _gpu_run(pr)
    pr0 = inputs.LoraProblem(pr.x, pr.W, pr.A, pr.B, torch.zeros_like(pr.gate), pr.alpha)
    y0 = _gpu_run(pr0)
    z = (pr.gate == 0).cuda()
    assert torch.equal(y[z].view(torch.int16), y0[z].view(torch.int16))
    assert not torch.equal(y[~z], y0[~z])


def test_rank_zero_and_alpha_zero():
    pr = inputs.lora_problem(24, 512, 256, 32, 64.0, name="r0")
    base = oracle.gated_lora_linear(pr.x, pr.W, pr.A, pr.B, torch.zeros_like(pr.gate), 0.0)
    pr_r0 = inputs.LoraProblem(pr.x, pr.W, pr.A[:0], pr.B[:, :0].contiguous(), pr.gate, pr.alpha)
    assert gemm_err(_gpu_run(pr_r0), base) <= GEMM_TOL
    pr_a0 = inputs.LoraProblem(pr.x, pr.W, pr.A, pr.B, pr.gate, 0.0)
    assert gemm_err(_gpu_run(pr_a0), base) <= GEMM_TOL


def test_deterministic():
    pr = inputs.lora_problem(32, 4096, 14336, 128, 256.0, name="det")
    a = _gpu_run(pr)
    b = _gpu_run(pr)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_no_device_error_flag():
    from lossless_draft_verify_gated_b300 import uno_device_error
    assert uno_device_error() == 0


def _batched(problems_pr, dtype=torch.bfloat16):
    from lossless_draft_verify_gated_b300 import uno_gated_lora_linear_batched
    d = "cuda"
    probs = []
    for pr in problems_pr:
        y = torch.empty((pr.x.shape[0], pr.W.shape[0]), dtype=dtype, device=d)
        probs.append((pr.x.to(d), pr.W.to(d), pr.A.to(d), pr.B.to(d), pr.gate.to(d), pr.alpha, y))
    ys = uno_gated_lora_linear_batched(probs)
    torch.cuda.synchronize()
    return ys


@pytest.mark.parametrize("M", [32, 16])
def test_batched_llama3_layer_decode(M):
    """All 7 projections of the Llama-3-8B-shaped layer in one persistent launch."""
    layer = inputs.llama3_layer(M, rank=128, alpha=256.0, block=16 if M >= 32 else 8)
    ys = _batched([pr for _, pr in layer])
    for (name, pr), y in zip(layer, ys):
        assert gemm_err(y, _ref(pr)) <= GEMM_TOL, name


def test_batched_llama3_layer_large_m_sampled():
    M = 2048
    layer = inputs.llama3_layer(M, rank=128, alpha=256.0, block=16)
    ys = _batched([pr for _, pr in layer])
    rows = torch.randperm(M, generator=inputs.generator("rows.batched"))[:32]
    for (name, pr), y in zip(layer, ys):
        assert gemm_err(y[rows.cuda()], _ref(pr, rows)) <= GEMM_TOL, name


@pytest.mark.parametrize("M", [24, 300])
def test_batched_mixed_ranks_and_shapes(M):
    """Rank 0 next to rank 8, 24 and 128, ragged d_in/d_out, swap and non-swap paths."""
    shapes = [(200, 136, 24, 48.0), (512, 1000, 0, 1.0), (64, 520, 128, 256.0), (1032, 72, 8, 16.0)]
    prs = [inputs.lora_problem(M, di, do, r, a, block=4, name=f"mix.{M}.{i}")
           for i, (di, do, r, a) in enumerate(shapes)]
    ys = _batched(prs)
    for pr, y in zip(prs, ys):
        assert gemm_err(y, _ref(pr)) <= GEMM_TOL


def test_batched_pair_order_mixed_ranks():
    """The pair order with ranks 0, 32, 64 and 128 in one launch (T tiles whose
    halves are 16, 32 and 64 output rows), ragged d_in and d_out, and a last
    problem whose trailing columns run as a 128-wide tile (8 real columns):
    64 seeded rows against the oracle over every column."""
    M = 2048
    shapes = [(512, 1000, 32, 64.0), (256, 520, 0, 1.0), (1024, 2048, 128, 256.0), (384, 264, 64, 128.0)]
    prs = [inputs.lora_problem(M, di, do, r, a, block=16, name=f"pairmix.{i}")
           for i, (di, do, r, a) in enumerate(shapes)]
    ys = _batched(prs)
    rows = torch.randperm(M, generator=inputs.generator("rows.pairmix"))[:64]
    for pr, y in zip(prs, ys):
        assert gemm_err(y[rows.cuda()], _ref(pr, rows)) <= GEMM_TOL
    from lossless_draft_verify_gated_b300 import uno_device_error
    assert uno_device_error() == 0


def test_batched_fp32():
    prs = [inputs.lora_problem(16, 256, 256, 16, 32.0, dtype=torch.float32, block=4, name=f"f32.{i}")
           for i in range(3)]
    ys = _batched(prs, dtype=torch.float32)
    for pr, y in zip(prs, ys):
        assert y.dtype == torch.float32
        assert gemm_err(y, _ref(pr)) <= GEMM_TOL


def test_batched_deterministic():
    layer = inputs.llama3_layer(32, seed=7)
    a = _batched([pr for _, pr in layer])
    b = _batched([pr for _, pr in layer])
    for ya, yb in zip(a, b):
        assert torch.equal(ya.view(torch.int16), yb.view(torch.int16))


LAYER_GROUPS = [["q", "k", "v"], ["o"], ["gate", "up"], ["down"]]


@pytest.mark.parametrize("M", [256, 512, 1024, 4096, 16384])
def test_layer_groups_sweep_sampled(M):
    """The layer's projections as the benchmark launches them (one grouped
    launch each for q/k/v, o, gate/up and down) at the row counts of the batch
    sweep (batch 8, 32, 128, 512 x 2 x block 16) and at batch 16 (q/k/v and
    gate/up in the pair order, gate/up with a 128-wide tail; o and down in
    token-rows stream-K):
    64 seeded rows, half gate 0 and half gate 1, against the oracle over every
    column."""
    layer = dict(inputs.llama3_layer(M, rank=128, alpha=256.0, block=16))
    g = inputs.generator(f"rows.sweep.{M}")
    perm = torch.randperm(M, generator=g)
    gate = layer["q"].gate
    rows = torch.cat([perm[gate[perm] == 0][:32], perm[gate[perm] == 1][:32]])
    for names in LAYER_GROUPS:
        ys = _batched([layer[n] for n in names])
        for n, y in zip(names, ys):
            assert gemm_err(y[rows.cuda()], _ref(layer[n], rows)) <= GEMM_TOL, (M, n)
        del ys
    from lossless_draft_verify_gated_b300 import uno_device_error
    assert uno_device_error() == 0
