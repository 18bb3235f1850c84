"""Host-side invariants of the projection kernel's schedule, checked on the
CPU through the library's own scheduler (uno_lora_plan_check, no GPU): the
grid fits one CTA per SM, each stream-K section's K-blocks are partitioned
over the CTAs in order, data-parallel waves cover every tile, a split T
tile's finisher takes no other work (decode order) or a split T tile's pieces
are whole ranges of consecutive CTAs (token-rows order), the workspace
regions fit.  The waits of the kernel end only if these hold (a split tile's
contributors are later CTAs, all resident at once)."""
import random

import pytest

from lossless_draft_verify_gated_b300 import binding

LLAMA_GROUPS = [[(4096, 4096, 128), (4096, 1024, 128), (4096, 1024, 128)], [(4096, 4096, 128)],
                [(4096, 14336, 128), (4096, 14336, 128)], [(14336, 4096, 128)]]
M_SWEEP = [1, 2, 8, 16, 31, 32, 48, 64, 100, 128, 129, 200, 255, 256, 512, 1024, 2048, 4096, 8192, 16384]


@pytest.mark.parametrize("sms", [148, 160, 132, 100, 37, 8, 1])
def test_llama_layer_groups(sms):
    for shapes in LLAMA_GROUPS:
        for M in M_SWEEP:
            for rank in (0, 16, 128):
                sh = [(di, do, rank) for di, do, _ in shapes]
                assert binding.uno_lora_plan_check(sh, M, sms) == 0, (sh, M, sms)


def test_random_shapes():
    rng = random.Random(2024)
    for _ in range(400):
        n = rng.randint(1, 8)
        sh = [(8 * rng.randint(1, 2500), 8 * rng.randint(1, 3600), 8 * rng.randint(0, 32))
              for _ in range(n)]
        M = rng.choice([rng.randint(1, 128), rng.randint(129, 6000)])
        sms = rng.choice([148, 148, 132, 64, 16, 3])
        dtype = rng.choice([0, 1])
        assert binding.uno_lora_plan_check(sh, M, sms, dtype) == 0, (sh, M, sms, dtype)


def test_refused_arguments():
    assert binding.uno_lora_plan_check([(12, 16, 8)], 32, 148) == -1   # d_in not a multiple of 8
    assert binding.uno_lora_plan_check([(16, 16, 264)], 32, 148) == -1  # rank above 256
    assert binding.uno_lora_plan_check([(16, 16, 8)], 32, 0) == -1      # no SMs
    assert binding.uno_lora_plan_check([(16, 16, 8)] * 9, 32, 148) == -1
