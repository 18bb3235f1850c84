"""bench.py's reference arm (the fp64 oracle on host cores) prints one JSON
line with the contract's keys, on the same workload as the GPU arm."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e", "gpu_launches"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["unit"] == "tokens/s" and d["steps"] == 1 and d["gpu_launches"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    sys.path.insert(0, ROOT)
    import bench
    assert d["config"]["workload"] == bench.workload_name(1)
    assert d["metric"] == bench.METRIC


def test_oracle_arms_draw_the_gpu_arms_verifier_sets():
    """The oracle's arms verify the input sets that the GPU arm's headline
    steps cycle through (set k drawn with the CPU generators from seed
    BASE_SEED + k, set 0 the one of the parity sample), and count tokens per
    step as the mean over those sets."""
    import torch
    sys.path.insert(0, ROOT)
    import bench
    from lossless_draft_verify_gated_b300 import inputs
    ob = bench.OracleStep(1, 1.0)
    assert ob.nsets == bench.n_verify_sets(1) == bench.VERIFY_SET_SEQS
    assert bench.n_verify_sets(8) == 8 and bench.n_verify_sets(512) == 1
    assert ob.vset(0)[0] is ob.vp
    vp3, draft3, _ = ob.vset(3)
    ref = inputs.verify_problem(1, bench.BLOCK, bench.VOCAB, sigma=1.0, seed=inputs.BASE_SEED + 3)
    assert torch.equal(vp3.p_logits, ref.p_logits) and torch.equal(vp3.u_resample, ref.u_resample)
    assert not torch.equal(vp3.p_logits, ob.vp.p_logits)
    assert draft3.shape == (1, bench.BLOCK)
    ob.nsets = 3  # the mean over the first three sets, verified one by one
    want = sum(float(ob.verify_sample(k).n_emitted.sum()) for k in range(3)) / 3
    assert ob.mean_tokens() == want


def test_end_to_end_steps_cover_the_timed_steps_sets():
    """The end-to-end figure verifies the sets of the K device-timed steps: all
    K of them up to one round of the sets, else whole rounds."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench.e2e_steps(20, 64) == 20
    assert bench.e2e_steps(64, 64) == 64
    assert bench.e2e_steps(2000, 64) == 64
    assert bench.e2e_steps(2000, 8) == 48
    assert bench.e2e_steps(2000, 1) == 50
    assert bench.e2e_steps(3, 1) == 3
