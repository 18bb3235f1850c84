"""Benchmark of one Uno draft+verify step on B300.

One step = the 7 gated-LoRA projections of one Llama-3-8B-shaped layer
(q 4096->4096, k/v 4096->1024, o 4096->4096, gate/up 4096->14336,
down 14336->4096; rank 128, alpha 256; M = 2*block*batch rows, half
verification rows with gate 0, half draft rows with gate 1), followed by the
block verifier over a 128256-entry vocabulary (batch x block 16, fp32 logits,
draft logits = AR logits + N(0, sigma)).  Inputs are seeded synthetic data
(inputs.py) resident in HBM; weights are random-init bf16.  The layer stands in
for a step (a full model would repeat the projections per layer).

Metric: verified tokens per second = sum over sequences of the tokens the
verifier emits in a step, divided by the device time of the step.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--batch B]
       python bench.py --impl reference ...   (the fp64 CPU oracle, timed)
Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified tokens/s per draft+verify step at batch 1–512; % of HBM/tensor roofline"
UNIT = "tokens/s"
BLOCK = 16
VOCAB = 128256
RANK = 128
ALPHA = 256.0
SIGMA = 1.0
L2_BYTES = 126 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--sigma", type=float, default=SIGMA)
    ap.add_argument("--impl", choices=["uno", "reference"], default="uno")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the batch sweep (batch 1-512) and the verifier sigma sweep")
    ap.add_argument("--sweep-steps", type=int, default=20, help="timed steps per sweep point")
    ap.add_argument("--no-graph", action="store_true", help="launch ops eagerly instead of replaying a CUDA graph")
    ap.add_argument("--temperature", type=float, default=1.0,
                    help="sampling temperature of the verifier (drafts drawn from q at the same T)")
    ap.add_argument("--resample", choices=["race", "inverse_cdf"], default="race",
                    help="residual/bonus draw: exponential race (default) or single-uniform inverse CDF")
    ap.add_argument("--grouping", choices=["layer", "all", "single"], default="layer",
                    help="layer: [q,k,v] [o] [gate,up] [down], one persistent launch each (the "
                         "layer's data dependencies); all: the 7 projections in one launch; "
                         "single: one launch per projection")
    return ap.parse_args()


def peaks():
    """(HBM GB/s, bf16 TFLOP/s burst, bf16 TFLOP/s sustained under the power cap, source)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        burst = float(p["bf16_tflops"])
        return float(p["hbm_gbs"]), burst, float(p.get("bf16_tflops_sustained", burst)), "measured"
    except Exception:
        return 6400.0, 1800.0, 1400.0, "fallback"


def kernel_source_hash():
    """sha256 (16 hex digits) of the projection kernel's sources with comments
    and whitespace removed: edits to the code invalidate recorded counters,
    edits to comments do not."""
    import hashlib
    import re
    h = hashlib.sha256()
    for name in ("gemm.cu", "ptx.cuh", "uno_internal.h"):
        with open(os.path.join(ROOT, "lossless_draft_verify_gated_b300", "csrc", name)) as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        h.update(re.sub(r"\s+", "", src).encode())
    return h.hexdigest()[:16]


def profiled_traffic(batch, launches):
    """DRAM bytes per projection launch from the committed ncu summary, or None
    when there is none for this workload or the kernel sources changed since."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"gemm_traffic_llama3_layer_b{batch}.txt")
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kernel_source_hash() != kv.get("source_sha256_16") or int(kv["launches_per_step"]) != launches:
            return None
        return int(kv["traffic_bytes_per_launch"])
    except Exception:
        return None


def workload_name(batch):
    return (f"llama3-8b-layer b{batch} k{BLOCK}: 7 gated-LoRA projections M={2 * BLOCK * batch} "
            f"r={RANK} alpha={int(ALPHA)} bf16 + block verifier B={batch} K={BLOCK} V={VOCAB} fp32")


def proj_bytes_flops(M, n_gate1):
    """Algorithmic HBM bytes and flops of the 7 projections: weights, adapters,
    activations in and out once; flops of the base GEMM on every row and of the
    adapter only on gate-1 rows."""
    from lossless_draft_verify_gated_b300 import inputs
    by = fl = 0
    for _, di, do in inputs.LLAMA3_8B_PROJECTIONS:
        by += 2 * (di * do + RANK * (di + do) + M * di + M * do)
        fl += 2 * M * di * do + 2 * n_gate1 * RANK * (di + do)
    return by, fl


def verify_bytes(batch, n_race, resample="race"):
    """p and q once, drafts and accept uniforms, and the resample's uniforms:
    a vocabulary row per race, one value per sequence for the inverse CDF."""
    u = 4 * VOCAB * n_race if resample == "race" else 4 * batch
    return 8 * batch * BLOCK * VOCAB + 12 * batch * BLOCK + u


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a run
    (started before the warm-up so that a short timed region is covered)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, period_ms=50):
        self.index = index
        self.period_ms = period_ms
        self.p = None
        self.out = ""

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.p is not None:
            self.p.terminate()
            try:
                self.out, _ = self.p.communicate(timeout=5)
            except Exception:
                self.p.kill()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 9:
                try:
                    rows.append((float(f[1]), float(f[2]), float(f[3]), f[5:9]))
                except ValueError:
                    pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        load = [r for r in rows if r[2] > 200.0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in load for n, v in zip(names, r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in load), "sm_max_mhz": max(r[1] for r in rows),
                "samples": len(load), "reasons": reasons}


def dist_setup(n_gpus):
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return ws, rank, local


def aggregate(ms_step, tokens, ws, device):
    """Whole-job figures over the ranks: the slowest rank's step time and the
    tokens every rank verified (each rank runs its own replica; this is the
    only exchange, host-side, outside the timed region)."""
    if ws == 1:
        return ms_step, tokens
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms_step], dtype=torch.float64, device=device)
    n = torch.tensor([tokens], dtype=torch.int64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), int(n.item())


GROUPINGS = {"layer": [["q", "k", "v"], ["o"], ["gate", "up"], ["down"]],
             "all": [["q", "k", "v", "o", "gate", "up", "down"]],
             "single": [["q"], ["k"], ["v"], ["o"], ["gate"], ["up"], ["down"]]}

SWEEP_BATCHES = (1, 8, 32, 128, 512)   # full step at batch 1-512 (M = 32 x batch)
SWEEP_SIGMAS = (0.25, 1.0, 4.0)        # verifier alone at batch 256, acceptance high to low
SWEEP_VERIFY_BATCH = 256


def config_dict(args, batch, ws):
    """The workload, identical in both arms (run details sit outside it)."""
    return {"workload": workload_name(batch), "batch": batch, "block": BLOCK, "vocab": VOCAB,
            "rank": RANK, "alpha": ALPHA, "sigma": args.sigma,
            "rows_per_projection": 2 * BLOCK * batch,
            "grouping": args.grouping + ": " + " | ".join(",".join(g) for g in GROUPINGS[args.grouping]),
            "sampler": f"temperature {args.temperature}, {args.resample} resample",
            "l2": "flushed before every step (2x L2 write, outside the timed events)",
            "parallelism": f"dp{ws} (independent replicas, no collective)"}


class Step:
    """All inputs, outputs and workspaces of one step, resident on the device.
    host_inputs: draw the seeded inputs with the CPU generators (the ones the
    oracle sample reads) and copy them over, instead of drawing on the device."""

    def __init__(self, batch, sigma, device, grouping="layer", temperature=1.0, resample="race",
                 host_inputs=False, with_layer=True):
        import torch
        from lossless_draft_verify_gated_b300 import binding, inputs
        self.batch, self.device = batch, device
        self.M = 2 * BLOCK * batch
        gen_dev = "cpu" if host_inputs else device
        self.groups = []
        self.layer = []
        if with_layer:
            self.layer = inputs.llama3_layer(self.M, rank=RANK, alpha=ALPHA, block=BLOCK, device=gen_dev)
            if host_inputs:
                moved = {}
                for _, pr in self.layer:
                    for f in ("x", "W", "A", "B", "gate"):
                        t = getattr(pr, f)
                        if t.data_ptr() not in moved:
                            moved[t.data_ptr()] = t.to(device)
                        setattr(pr, f, moved[t.data_ptr()])
            by_name = dict(self.layer)
            self.ys = {n: torch.empty((self.M, p.W.shape[0]), dtype=torch.bfloat16, device=device)
                       for n, p in self.layer}
            for names in GROUPINGS[grouping]:
                probs = [(by_name[n].x, by_name[n].W, by_name[n].A, by_name[n].B, by_name[n].gate,
                          by_name[n].alpha, self.ys[n]) for n in names]
                shapes = [(p[0].shape[1], p[1].shape[0], p[2].shape[0]) for p in probs]
                ws = torch.empty(binding.uno_gated_lora_linear_batched_workspace(shapes, self.M, 1),
                                 dtype=torch.uint8, device=device)
                self.groups.append((probs, ws))
            self.n_gate1 = int(self.layer[0][1].gate.sum())
        vp = inputs.verify_problem(batch, BLOCK, VOCAB, sigma=sigma, device=gen_dev)
        if host_inputs:
            vp = inputs.VerifyProblem(*(t.to(device) for t in (vp.p_logits, vp.q_logits, vp.u_accept,
                                                               vp.u_resample, vp.u_draft)))
        self.p, self.q, self.ua, self.ur = vp.p_logits, vp.q_logits, vp.u_accept, vp.u_resample
        self.temperature, self.resample = temperature, resample
        self.plain = temperature == 1.0 and resample == "race"
        if resample == "inverse_cdf":  # one uniform per sequence
            self.ur = inputs.uniform_accept((batch,), f"verify.u1.B{batch}", device=device)
        # drafts: the linear sampler's drafting half, a single token drawn from q (at the
        # verifier's temperature) at each position
        qd = self.q if temperature == 1.0 else (self.q.double() / temperature).float()
        self.draft, st = binding.uno_draft_sample(qd, vp.u_draft)
        del qd
        assert int(st.abs().sum()) == 0
        del vp
        self.vout = tuple(torch.empty(s, dtype=torch.int32, device=device)
                          for s in [(batch,), (batch, BLOCK + 1), (batch,), (batch,)])
        self.vws = torch.empty(binding.uno_verify_block_workspace(batch, BLOCK, BLOCK, VOCAB),
                               dtype=torch.uint8, device=device)
        # kernels of this library per step: per group a one-CTA flag reset and the
        # persistent GEMM, then the verifier's two kernels
        self.launches_per_step = 2 * len(self.groups) + 2

    def projections(self):
        from lossless_draft_verify_gated_b300 import binding
        for probs, ws in self.groups:
            binding.uno_gated_lora_linear_batched(probs, workspace=ws)

    def verify(self):
        from lossless_draft_verify_gated_b300 import binding
        if self.plain:
            binding.uno_verify_block(self.p, self.q, self.draft, self.ua, self.ur, out=self.vout,
                                     workspace=self.vws)
        else:
            binding.uno_verify_block_ex(self.p, self.q, self.draft, self.ua, self.ur,
                                        temperature=self.temperature, resample=self.resample,
                                        out=self.vout, workspace=self.vws)


class Timer:
    """Replays the two halves of a step (projections, verifier) from CUDA graphs
    and times each half with CUDA events on the launching stream, with an L2
    flush (a write of twice the L2 size) before every step outside the events."""

    def __init__(self, st, dev, graph=True):
        import torch
        self.st = st
        self.flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
        self.g_proj = self.g_ver = None
        if graph:
            s = torch.cuda.Stream(device=dev)
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                st.projections()
                st.verify()
            torch.cuda.current_stream().wait_stream(s)
            torch.cuda.synchronize()
            self.g_proj = torch.cuda.CUDAGraph() if st.groups else None
            self.g_ver = torch.cuda.CUDAGraph()
            if self.g_proj is not None:
                with torch.cuda.graph(self.g_proj):
                    st.projections()
            with torch.cuda.graph(self.g_ver):
                st.verify()

    def proj(self):
        if self.g_proj is not None:
            self.g_proj.replay()
        elif self.st.groups:
            self.st.projections()

    def ver(self):
        self.g_ver.replay() if self.g_ver is not None else self.st.verify()

    def warm(self, n):
        import torch
        for _ in range(n):
            self.flush.zero_()
            self.proj()
            self.ver()
        torch.cuda.synchronize()

    def run(self, steps, barrier=None):
        """Per-step (step, projections, verifier) milliseconds and the wall time."""
        import torch
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        if barrier:
            barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(steps):
            self.flush.zero_()  # L2 flush, outside the timed events
            ev[i][0].record()
            self.proj()
            ev[i][1].record()
            self.ver()
            ev[i][2].record()
        torch.cuda.synchronize()
        if barrier:
            barrier()
        wall = time.perf_counter() - t0
        return ([e[0].elapsed_time(e[2]) for e in ev], [e[0].elapsed_time(e[1]) for e in ev],
                [e[1].elapsed_time(e[2]) for e in ev], wall)


def proj_roofline(M, n_gate1, ms_proj, hbm, tflops):
    """Bound, achieved, peak and unit of the layer's projections."""
    by, fl = proj_bytes_flops(M, n_gate1)
    bound = "hbm" if fl / by < (tflops * 1e12) / (hbm * 1e9) else "tensor"
    if bound == "hbm":
        return bound, by / (ms_proj / 1e3) / 1e9, hbm, "GB/s", by, fl
    return bound, fl / (ms_proj / 1e3) / 1e12, tflops, "TFLOP/s", by, fl


def check_device_error():
    from lossless_draft_verify_gated_b300 import binding
    err = binding.uno_device_error()
    if err != 0:
        raise RuntimeError(f"projection kernel reported device error word {err}: outputs invalid")
    return err


def sweep(args, dev, hbm, tflops, tflops_sustained):
    """Config 5 (the whole step at batch 1-512) and config 4 (the verifier alone
    at batch 256 for three draft-noise levels), each point timed like the
    headline on its own device-drawn seeded inputs."""
    import torch
    out = {"steps_per_point": args.sweep_steps, "warmup_per_point": 3, "step": [], "verifier_sigma": []}
    for b in SWEEP_BATCHES:
        st = Step(b, SIGMA, dev, args.grouping)
        tm = Timer(st, dev)
        tm.warm(3)
        t_step, t_proj, t_ver, _ = tm.run(args.sweep_steps)
        check_device_error()
        n_acc, _, n_em, vstat = (t.cpu() for t in st.vout)
        assert int(vstat.abs().sum()) == 0
        ms_step, ms_proj, ms_ver = (statistics.mean(t) for t in (t_step, t_proj, t_ver))
        bound, ach, peak, unit, _, _ = proj_roofline(st.M, st.n_gate1, ms_proj, hbm, tflops)
        vb = verify_bytes(b, int((n_acc < BLOCK).sum()))
        e = {"batch": b, "rows_per_projection": st.M, "ms_per_step": round(ms_step, 5),
             "tokens_per_s": round(int(n_em.sum()) / (ms_step / 1e3), 1),
             "verified_tokens_per_step": int(n_em.sum()),
             "projections": {"ms": round(ms_proj, 5), "bound": bound, "achieved": round(ach, 2),
                             "unit": unit, "frac": round(ach / peak, 4)},
             "verifier": {"ms": round(ms_ver, 5), "bytes": vb,
                          "frac_hbm": round(vb / (ms_ver / 1e3) / 1e9 / hbm, 4)}}
        if bound == "tensor":
            e["projections"]["frac_of_sustained"] = round(ach / tflops_sustained, 4)
        out["step"].append(e)
        del tm, st
        torch.cuda.empty_cache()
    for sg in SWEEP_SIGMAS:
        b = SWEEP_VERIFY_BATCH
        st = Step(b, sg, dev, with_layer=False)
        tm = Timer(st, dev)
        tm.warm(3)
        _, _, t_ver, _ = tm.run(args.sweep_steps)
        n_acc, _, n_em, vstat = (t.cpu() for t in st.vout)
        assert int(vstat.abs().sum()) == 0
        ms_ver = statistics.mean(t_ver)
        vb = verify_bytes(b, int((n_acc < BLOCK).sum()))
        out["verifier_sigma"].append({
            "batch": b, "sigma": sg, "ms": round(ms_ver, 5),
            "tokens_per_s": round(int(n_em.sum()) / (ms_ver / 1e3), 1),
            "mean_accepted": round(float(n_acc.float().mean()), 3),
            "mean_emitted": round(float(n_em.float().mean()), 3),
            "bytes": vb, "frac_hbm": round(vb / (ms_ver / 1e3) / 1e9 / hbm, 4)})
        del tm, st
        torch.cuda.empty_cache()
    return out


def run_uno(args):
    import torch
    ws, rank, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    from lossless_draft_verify_gated_b300 import binding
    binding.lib()
    hbm, tflops, tflops_sustained, peak_kind = peaks()
    # The headline step at N=1 reads the CPU-drawn inputs that the oracle sample
    # reads too, so that its outputs can be compared with the oracle's.
    check_parity = rank == 0 and ws == 1 and not args.no_cpu_baseline and args.temperature == 1.0 \
        and args.resample == "race" and args.batch <= 8
    st = Step(args.batch, args.sigma, dev, args.grouping, args.temperature, args.resample,
              host_inputs=check_parity)
    K = args.steps
    with Clocks(local) as clk:
        tm = Timer(st, dev, graph=not args.no_graph)
        tm.warm(args.warmup)
        check_device_error()
        barrier = torch.distributed.barrier if ws > 1 else None
        t_step, t_proj, t_ver, wall = tm.run(K, barrier)
    device_error = check_device_error()
    n_acc, toks, n_em, vstat = (t.cpu() for t in st.vout)
    assert int(vstat.abs().sum()) == 0
    ms_step, tokens_all = aggregate(sum(t_step) / K, int(n_em.sum()), ws, dev)
    tokens = tokens_all // ws  # per replica (every replica runs the same seeded step)
    value = tokens_all / (ms_step / 1e3)

    # roofline of the dominant op: the layer's gated-LoRA projections
    ms_proj = statistics.mean(t_proj)
    ms_ver = statistics.mean(t_ver)
    bound, achieved, peak, unit, by, fl = proj_roofline(st.M, st.n_gate1, ms_proj, hbm, tflops)
    n_race = int((n_acc < BLOCK).sum())
    vb = verify_bytes(args.batch, n_race, args.resample)
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_dict(args, args.batch, ws),
        "verified_tokens_per_step": tokens,
        "launch": "CUDA graph per half-step" if tm.g_ver is not None else "eager",
        "inputs": "CPU-drawn seeded inputs copied to the device" if check_parity else
                  "seeded inputs drawn on the device",
        "roofline": {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
                     "frac": round(achieved / peak, 4),
                     "traffic": profiled_traffic(args.batch, len(st.groups)),
                     "algorithmic_bytes_per_launch": by // len(st.groups),
                     "kernel": f"gated-LoRA projections of the layer ({len(st.groups)} persistent grouped GEMM launch(es))",
                     "peak_source": peak_kind, "algorithmic_bytes": by, "algorithmic_flops": fl,
                     "ms": round(ms_proj, 5)},
        "verifier": {"ms": round(ms_ver, 5), "bytes": vb,
                     "achieved_gbs": round(vb / (ms_ver / 1e3) / 1e9, 2),
                     "frac_hbm": round(vb / (ms_ver / 1e3) / 1e9 / hbm, 4)},
        "gpu_launches": st.launches_per_step * K,
        "device_error": device_error,
        "wall_s": round(wall, 3),
    }
    if bound == "tensor":
        # The step's projections run back to back for the whole timed region: under the
        # 1.1 kW cap the clocks settle (sw_power_cap), as in the sustained GEMM measurement.
        out["roofline"]["peak_sustained"] = tflops_sustained
        out["roofline"]["frac_of_sustained"] = round(achieved / tflops_sustained, 4)
    out["clocks"] = clk.summary()
    if not args.no_e2e:
        out["e2e"] = e2e(st, dev, max(5, min(K, 50)), ws)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        if st.plain:
            out["cpu_baseline"] = cpu_baseline(st, args.batch, args.sigma, budget_s=15.0,
                                               compare=check_parity)
        else:  # the timed oracle step is the default sampler's
            out["cpu_baseline"] = None
    del tm, st
    torch.cuda.empty_cache()
    if rank == 0 and ws == 1 and not args.no_sweep and args.temperature == 1.0 and args.resample == "race":
        with Clocks(local) as clk2:
            out["sweep"] = sweep(args, dev, hbm, tflops, tflops_sustained)
        out["sweep"]["clocks"] = clk2.summary()
    if rank == 0:
        print(json.dumps(out), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def e2e(st, dev, steps, ws=1):
    """Same metric through the public API with host buffers: every step copies
    its inputs host->device from pinned memory, runs the ops eagerly and reads
    the verified tokens back.  Also reported: the time of the copies alone and
    the host time spent in the API calls (enqueue, no synchronisation)."""
    import torch
    host = {}
    seen = set()
    for i, (_, p) in enumerate(st.layer):
        for tag, t in (("x", p.x), ("g", p.gate)):
            if t.data_ptr() not in seen:  # q/k/v and gate/up share their input; one gate tensor
                seen.add(t.data_ptr())
                host[f"{tag}{i}"] = (t.cpu().pin_memory(), t)
    for k in ("p", "q", "draft", "ua", "ur"):
        t = getattr(st, k)
        host[k] = (t.cpu().pin_memory(), t)
    h2d = sum(h.numel() * h.element_size() for h, _ in host.values())
    outs = [torch.empty_like(st.vout[1], device="cpu").pin_memory(),
            torch.empty_like(st.vout[2], device="cpu").pin_memory()]
    d2h = sum(o.numel() * o.element_size() for o in outs)
    torch.cuda.synchronize()

    def copies():
        for h, d in host.values():
            d.copy_(h, non_blocking=True)

    def one():
        copies()
        st.projections()
        st.verify()
        outs[0].copy_(st.vout[1], non_blocking=True)
        outs[1].copy_(st.vout[2], non_blocking=True)

    for _ in range(3):
        one()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # the copies alone
    e0.record()
    for _ in range(steps):
        copies()
    e1.record()
    torch.cuda.synchronize()
    ms_copy = e0.elapsed_time(e1) / steps
    # host time of the API calls alone (enqueue only)
    t_api = 0.0
    for _ in range(steps):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        st.projections()
        st.verify()
        t_api += time.perf_counter() - t0
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    e0.record()
    for _ in range(steps):
        one()
    e1.record()
    torch.cuda.synchronize()
    check_device_error()
    ms, tokens = aggregate(e0.elapsed_time(e1) / steps, int(outs[1].sum()), ws, dev)
    return {"value": round(tokens / (ms / 1e3), 2), "unit": UNIT, "ms_per_step": round(ms, 4),
            "steps": steps, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "h2d_ms_per_step": round(ms_copy, 4), "host_api_ms_per_step": round(t_api / steps * 1e3, 4),
            "launch": "eager API calls"}


def cpu_inputs(batch, sigma):
    """The same workload drawn on the host (CPU generators), drafts drawn by
    the oracle's own sampler."""
    from lossless_draft_verify_gated_b300 import inputs
    import oracle
    M = 2 * BLOCK * batch
    layer = inputs.llama3_layer(M, rank=RANK, alpha=ALPHA, block=BLOCK)
    vp = inputs.verify_problem(batch, BLOCK, VOCAB, sigma=sigma)
    draft, _, margin = oracle.draft_sample(vp.q_logits, vp.u_draft)
    return layer, vp, draft.reshape(batch, BLOCK), margin.reshape(batch, BLOCK)


class OracleStep:
    """The fp64 oracle as it stands, run on a bounded sample of one step and
    scaled to a full step.  Rows and output columns of a projection are
    independent, and so are sequences of the verifier, so the time of the
    sample scales by (rows x columns) and by sequences."""

    def __init__(self, batch, sigma):
        import oracle
        oracle.build()
        self.batch = batch
        self.M = 2 * BLOCK * batch
        self.layer, self.vp, self.draft, self.draft_margin = cpu_inputs(batch, sigma)
        self.threads = oracle.num_threads()
        self.rows = min(self.M, max(2, self.threads))
        self.seqs = min(batch, max(1, self.threads))
        self.col_frac = 1.0
        self.repeat = 1  # samples per timed step (a small step is repeated to time it reliably)
        self.last = None

    def row_index(self):
        import numpy as np
        M, rows = self.M, self.rows
        return np.concatenate([np.arange(rows // 2), M - 1 - np.arange(rows - rows // 2)])

    def run(self):
        import oracle
        M, rows = self.M, self.rows
        r_idx = self.row_index()
        tp = tv = 0.0
        ys = []
        for _ in range(self.repeat):
            t0 = time.perf_counter()
            scale_p = 0.0
            ys = []
            for name, p in self.layer:
                d_out = p.W.shape[0]
                c = max(8, int(round(d_out * self.col_frac / 8)) * 8)
                c = min(c, d_out)
                y = oracle.gated_lora_linear(p.x[r_idx], p.W[:c], p.A, p.B[:c], p.gate[r_idx], p.alpha)
                ys.append((name, c, y))
                scale_p = (M / rows) * (d_out / c)  # equal fractions for every projection
            t1 = time.perf_counter()
            s = self.seqs
            vp = self.vp
            r = oracle.verify_block(vp.p_logits[:s], vp.q_logits[:s], self.draft[:s], vp.u_accept[:s],
                                    vp.u_resample[:s])
            t2 = time.perf_counter()
            tp += t1 - t0
            tv += t2 - t1
        self.last = (r_idx, ys, r)
        t_full = (tp * scale_p + tv * (self.batch / s)) / self.repeat
        tokens = float(r.n_emitted.sum()) * (self.batch / s)
        return t_full, tokens, tp + tv

    def calibrate(self, target_s):
        """Pick the column fraction (and, when the whole step is shorter than
        target_s, a repeat count) so that one timed sample takes about target_s."""
        self.col_frac, self.repeat = 1.0 / 16, 1
        _, _, t = self.run()
        want = self.col_frac * target_s / max(t, 1e-3)
        self.col_frac = min(1.0, max(1.0 / 512, want))
        if want > 1.0:  # the whole step is short: time it once and repeat it
            _, _, t1 = self.run()
            self.repeat = max(1, min(1000, int(round(target_s / max(t1, 1e-3)))))

    def describe(self, steps):
        return (f"{self.rows} of {self.M} rows x {self.col_frac:.4f} of the output columns of each of "
                f"the 7 projections + the verifier for {self.seqs} of {self.batch} sequences per step, "
                f"scaled to the full step, each sample run {self.repeat}x and averaged; {steps} step(s)")

    def compare(self, st):
        """The GPU step's outputs on the sampled rows, columns and sequences
        against the oracle's: projections within 2e-2 x rms, verifier outputs
        bit-exact outside fp64 near-ties (margin < 1e-4); the drafts, which each
        side draws with its own sampler, must agree first."""
        import numpy as np
        import torch
        r_idx, ys, r = self.last
        worst = 0.0
        for name, c, y_ref in ys:
            rows = torch.as_tensor(r_idx, device=st.ys[name].device)
            y = st.ys[name][rows][:, :c].float().cpu().double().numpy()
            rms = float(np.sqrt(np.mean(y_ref ** 2)))
            worst = max(worst, float(np.abs(y - y_ref).max()) / rms)
        s = self.seqs
        g_draft = st.draft[:s].cpu().numpy()
        draft_tie = (self.draft_margin[:s] < 1e-4).any(axis=1)
        same_draft = (g_draft == self.draft[:s]).all(axis=1) | draft_tie
        keep = ~r.near_tie(1e-4) & ~draft_tie
        n_acc, toks, n_em, stt = (t[:s].cpu().numpy() for t in st.vout)
        ok_v = bool(same_draft.all() and (stt == r.status).all()
                    and (n_acc[keep] == r.n_accepted[keep]).all()
                    and (toks[keep] == r.out_tokens[keep]).all()
                    and (n_em[keep] == r.n_emitted[keep]).all())
        return {"ok": bool(worst <= 2e-2 and ok_v),
                "projections_max_err_over_rms": round(worst, 6), "projections_tolerance": 2e-2,
                "verifier_sequences": int(s), "verifier_excluded_near_ties": int((~keep).sum()),
                "verifier_bit_exact": ok_v}


def cpu_baseline(st, batch, sigma, budget_s=15.0, compare=False):
    ob = OracleStep(batch, sigma)
    ob.calibrate(budget_s)
    t_full, tokens, t_cpu = ob.run()
    out = {"value": round(tokens / t_full, 4), "unit": UNIT, "cores": ob.threads, "kind": "oracle",
           "sample": ob.describe(1) + f"; {t_cpu:.1f} s of CPU work",
           "ms_per_step_extrapolated": round(t_full * 1e3, 2)}
    if compare:
        out["parity"] = ob.compare(st)
    return out


def run_reference(args):
    """The oracle as the reference arm: each step runs the oracle on a bounded
    sample of the step (scaled to a full step) on the host cores, sized so the
    whole run stays within about two minutes."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    ob = OracleStep(args.batch, args.sigma)
    ob.calibrate(min(1.0, 120.0 / max(1, args.steps + args.warmup)))
    times, toks = [], []
    for i in range(args.warmup + args.steps):
        t_full, tokens, _ = ob.run()
        if i >= args.warmup:
            times.append(t_full)
            toks.append(tokens)
    ms = statistics.mean(times) * 1e3
    value = statistics.mean(toks) / (ms / 1e3)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": config_dict(args, args.batch, ws),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": ob.threads, "kind": "oracle",
                         "sample": ob.describe(args.steps)},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_uno(args)


if __name__ == "__main__":
    main()
