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
    ap.add_argument("--profile", choices=["lm_head", "tree"], default=None,
                    help="replay one op a few times for a profiler (no JSON line): the LM head + "
                         "verifier (--batch, --lm-mode) or the tree sampler (--batch)")
    ap.add_argument("--lm-mode", choices=["plain", "stats_store", "stats_recompute"], default="stats_recompute")
    ap.add_argument("--l2-flush", choices=["write", "write_read"], default="write_read",
                    help="L2 flush before every step, outside the timed events: a write of twice "
                         "the L2 size, then (write_read) a read of another such buffer, so that the "
                         "step does not start by writing back the flush's own dirty lines")
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
    return int(round(8 * batch * BLOCK * VOCAB + 12 * batch * BLOCK + u))


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
    n = torch.tensor([tokens], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), float(n.item())


GROUPINGS = {"layer": [["q", "k", "v"], ["o"], ["gate", "up"], ["down"]],
             "all": [["q", "k", "v", "o", "gate", "up", "down"]],
             "single": [["q"], ["k"], ["v"], ["o"], ["gate"], ["up"], ["down"]]}

SWEEP_BATCHES = (1, 8, 32, 128, 512)   # full step at batch 1-512 (M = 32 x batch)
SWEEP_SIGMAS = (0.25, 1.0, 4.0)        # verifier alone at batch 256, acceptance high to low
SWEEP_VERIFY_BATCH = 256
VERIFY_SET_SEQS = 64                   # a step at batch B cycles through 64 // B verifier input sets
LM_D = 4096                            # Llama-3-8B hidden size: the LM head is [128256, 4096]
SWEEP_LM_BATCHES = (1, 256)
SWEEP_TREE = ((1, (3, 2, 2, 1)), (8, (3, 2, 2, 1)))  # (batch, children per node at each depth)


def n_verify_sets(batch):
    """Verifier input sets that consecutive steps cycle through (step i verifies
    set i mod n, in every arm and in the end-to-end figure)."""
    return max(1, VERIFY_SET_SEQS // batch)


def config_dict(args, batch, ws):
    """The workload, identical in both arms (run details sit outside it)."""
    return {"workload": workload_name(batch), "batch": batch, "block": BLOCK, "vocab": VOCAB,
            "rank": RANK, "alpha": ALPHA, "sigma": args.sigma,
            "rows_per_projection": 2 * BLOCK * batch,
            "grouping": args.grouping + ": " + " | ".join(",".join(g) for g in GROUPINGS[args.grouping]),
            "sampler": f"temperature {args.temperature}, {args.resample} resample",
            "l2": ("flushed before every step, outside the timed events: a 2x L2 write" +
                   (", then a 2x L2 read of another buffer" if args.l2_flush == "write_read" else "")),
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
        self.temperature, self.resample = temperature, resample
        self.plain = temperature == 1.0 and resample == "race"
        # Verifier inputs: at a small batch the accepted lengths of a single draw
        # say little about the mean, so consecutive steps cycle through several
        # seeded input sets (at least VERIFY_SET_SEQS sequences in all), every
        # one drawn as host_inputs asks (with the CPU generators, the oracle's
        # arms draw the same sets).
        self.vsets = []
        for k in range(n_verify_sets(batch)):
            vp = inputs.verify_problem(batch, BLOCK, VOCAB, sigma=sigma, device=gen_dev,
                                       seed=inputs.BASE_SEED + k)
            if vp.p_logits.device != torch.device(device):
                vp = inputs.VerifyProblem(*(t.to(device) for t in (vp.p_logits, vp.q_logits, vp.u_accept,
                                                                   vp.u_resample, vp.u_draft)))
            ur = vp.u_resample
            if resample == "inverse_cdf":  # one uniform per sequence
                ur = inputs.uniform_accept((batch,), f"verify.u1.B{batch}.{k}", device=device)
            # drafts: the linear sampler's drafting half, a single token drawn from q
            # (at the verifier's temperature) at each position
            qd = vp.q_logits if temperature == 1.0 else (vp.q_logits.double() / temperature).float()
            draft, dst = binding.uno_draft_sample(qd, vp.u_draft)
            del qd
            assert int(dst.abs().sum()) == 0
            vout = tuple(torch.empty(sh, dtype=torch.int32, device=device)
                         for sh in [(batch,), (batch, BLOCK + 1), (batch,), (batch,)])
            self.vsets.append({"p": vp.p_logits, "q": vp.q_logits, "ua": vp.u_accept, "ur": ur,
                               "draft": draft, "vout": vout})
            del vp
        s0 = self.vsets[0]
        self.p, self.q, self.ua, self.ur, self.draft, self.vout = (s0[k] for k in
                                                                   ("p", "q", "ua", "ur", "draft", "vout"))
        self.vws = torch.empty(binding.uno_verify_block_workspace(batch, BLOCK, BLOCK, VOCAB),
                               dtype=torch.uint8, device=device)
        # kernels of this library per step: per group a one-CTA flag reset and the
        # persistent GEMM, then the verifier's two kernels
        self.launches_per_step = 2 * len(self.groups) + 2

    def projections(self):
        from lossless_draft_verify_gated_b300 import binding
        for probs, ws in self.groups:
            binding.uno_gated_lora_linear_batched(probs, workspace=ws)

    def verify(self, k=0):
        """The verifier on input set k."""
        from lossless_draft_verify_gated_b300 import binding
        v = self.vsets[k]
        if self.plain:
            binding.uno_verify_block(v["p"], v["q"], v["draft"], v["ua"], v["ur"], out=v["vout"],
                                     workspace=self.vws)
        else:
            binding.uno_verify_block_ex(v["p"], v["q"], v["draft"], v["ua"], v["ur"],
                                        temperature=self.temperature, resample=self.resample,
                                        out=v["vout"], workspace=self.vws)

    def set_of_step(self, i):
        return i % len(self.vsets)

    def verify_results(self, steps):
        """Host copies of every set's outputs and the tokens verified over
        `steps` steps (step i verified set i mod the number of sets)."""
        res = [tuple(t.cpu() for t in v["vout"]) for v in self.vsets]
        tokens = sum(int(res[self.set_of_step(i)][2].sum()) for i in range(steps))
        return res, tokens


class Timer:
    """Replays a step from CUDA graphs and times it with CUDA events on the
    launching stream, with an L2 flush before every step outside the events.
    The step is one graph (projections then verifier, chained as a serving
    loop would launch them); each half is also timed alone, from a graph of its
    own, for the projections' roofline and the verifier's fields."""

    def __init__(self, st, dev, graph=True, l2_flush="write_read"):
        import torch
        self.st = st
        self.flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
        self.flush_read = (torch.zeros(2 * L2_BYTES // 4, dtype=torch.int32, device=dev)
                           if l2_flush == "write_read" else None)
        self.g_proj = self.g_ver = None
        self.g_step = []
        if graph:
            s = torch.cuda.Stream(device=dev)
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                st.projections()
                st.verify()
            torch.cuda.current_stream().wait_stream(s)
            torch.cuda.synchronize()
            self.g_proj = torch.cuda.CUDAGraph() if st.groups else None
            if self.g_proj is not None:
                with torch.cuda.graph(self.g_proj):
                    st.projections()
            self.g_ver = []
            for k in range(len(st.vsets)):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    st.verify(k)
                self.g_ver.append(g)
            self.g_step = []
            if st.groups:
                for k in range(len(st.vsets)):
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g):
                        st.projections()
                        st.verify(k)
                    self.g_step.append(g)

    def proj(self):
        if self.g_proj is not None:
            self.g_proj.replay()
        elif self.st.groups:
            self.st.projections()

    def ver(self, i=0):
        k = self.st.set_of_step(i)
        self.g_ver[k].replay() if self.g_ver is not None else self.st.verify(k)

    def flush(self):
        """Evicts the step's inputs from L2: a write of twice its size, then
        (write_read) a read of another such buffer, leaving clean lines."""
        self.flush_buf.zero_()
        if self.flush_read is not None:
            self.flush_read.max()

    def warm(self, n):
        import torch
        for i in range(n):
            self.flush()
            self.proj()
            self.ver(i)
            if self.g_step:
                self.flush()
                self.g_step[self.st.set_of_step(i)].replay()
        torch.cuda.synchronize()

    def run(self, steps, barrier=None):
        """Per-step (step, projections, verifier) milliseconds and the wall
        time of the step's timed region.  With graphs, the step times come from
        the one-graph steps (the timed region the wall time covers); the two
        halves are then timed alone over as many steps again."""
        import torch
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        whole = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        if barrier:
            barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        if self.g_step:
            for i in range(steps):
                self.flush()  # L2 flush, outside the timed events
                whole[i][0].record()
                self.g_step[self.st.set_of_step(i)].replay()
                whole[i][1].record()
        else:
            for i in range(steps):
                self.flush()
                ev[i][0].record()
                self.proj()
                ev[i][1].record()
                self.ver(i)
                ev[i][2].record()
        torch.cuda.synchronize()
        if barrier:
            barrier()
        wall = time.perf_counter() - t0
        if self.g_step:
            for i in range(steps):
                self.flush()
                ev[i][0].record()
                self.proj()
                ev[i][1].record()
                self.ver(i)
                ev[i][2].record()
            torch.cuda.synchronize()
            t_step = [w[0].elapsed_time(w[1]) for w in whole]
        else:
            t_step = [e[0].elapsed_time(e[2]) for e in ev]
        return (t_step, [e[0].elapsed_time(e[1]) for e in ev], [e[1].elapsed_time(e[2]) for e in ev], wall)


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
        tm = Timer(st, dev, l2_flush=args.l2_flush)
        tm.warm(3)
        t_step, t_proj, t_ver, _ = tm.run(args.sweep_steps)
        check_device_error()
        res, tokens = st.verify_results(args.sweep_steps)
        assert all(int(r[3].abs().sum()) == 0 for r in res)
        ms_step, ms_proj, ms_ver = (statistics.mean(t) for t in (t_step, t_proj, t_ver))
        bound, ach, peak, unit, _, _ = proj_roofline(st.M, st.n_gate1, ms_proj, hbm, tflops)
        vb = verify_bytes(b, statistics.mean(int((r[0] < BLOCK).sum()) for r in res))
        per_step = tokens / args.sweep_steps
        e = {"batch": b, "rows_per_projection": st.M, "ms_per_step": round(ms_step, 5),
             "tokens_per_s": round(per_step / (ms_step / 1e3), 1),
             "verified_tokens_per_step": round(per_step, 3), "verifier_input_sets": len(st.vsets),
             "projections": {"ms": round(ms_proj, 5), "bound": bound, "achieved": round(ach, 2),
                             "unit": unit, "frac": round(ach / peak, 4)},
             "verifier": {"ms": round(ms_ver, 5), "bytes": vb,
                          "frac_hbm": round(vb / (ms_ver / 1e3) / 1e9 / hbm, 4)}}
        if bound == "tensor":
            e["projections"]["frac_of_sustained"] = round(ach / tflops_sustained, 4)
        out["step"].append(e)
        del tm, st
        torch.cuda.empty_cache()
    out["lm_head"] = lm_head_sweep(args, dev, hbm, tflops)
    out["tree"] = tree_sweep(args, dev, hbm)
    for sg in SWEEP_SIGMAS:
        b = SWEEP_VERIFY_BATCH
        st = Step(b, sg, dev, with_layer=False)
        tm = Timer(st, dev, l2_flush=args.l2_flush)
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


def make_flusher(dev, mode):
    """The L2 flush of --l2-flush as a callable (write, then optionally read)."""
    import torch
    wbuf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    rbuf = torch.zeros(2 * L2_BYTES // 4, dtype=torch.int32, device=dev) if mode == "write_read" else None

    def flush():
        wbuf.zero_()
        if rbuf is not None:
            rbuf.max()
    return flush


def time_graph(fn, steps, flush):
    """Median device time (ms) of fn replayed from a CUDA graph, L2 flushed
    (flush()) before each replay outside the timed events."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    ts = []
    for _ in range(3 + steps):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts[3:])


def lm_head_sweep(args, dev, hbm, tflops):
    """The LM head feeding the verifier (Llama-3-8B head [128256, 4096], block
    16, synthetic hidden states) in each of its three strategies: the logits
    stored and verified, the verifier's statistics taken in the GEMM's
    epilogue with the logits stored, and with only the resampled rows
    recomputed (no logit written).  logit_bytes = the logit traffic the
    strategy implies (written and read back)."""
    import torch
    from lossless_draft_verify_gated_b300 import binding, inputs
    flush = make_flusher(dev, args.l2_flush)
    res = []
    for b in SWEEP_LM_BATCHES:
        pr = inputs.lm_head_problem(b, BLOCK, VOCAB, LM_D, device=dev)
        W = pr.W
        qlog = torch.matmul(pr.h[b * BLOCK:].float(), W.float().T).reshape(b, BLOCK, VOCAB)
        draft, st = binding.uno_draft_sample(qlog, pr.u_draft)
        del qlog
        rows = 2 * BLOCK * b
        flops = 2.0 * rows * LM_D * VOCAB
        outs = {}
        for mode in ("plain", "stats_store", "stats_recompute"):
            ws = torch.empty(binding.uno_lm_head_verify_workspace(b, BLOCK, BLOCK, VOCAB, LM_D, mode),
                             dtype=torch.uint8, device=dev)
            out = tuple(torch.empty(sh, dtype=torch.int32, device=dev)
                        for sh in [(b,), (b, BLOCK + 1), (b,), (b,)])
            ms = time_graph(lambda: binding.uno_lm_head_verify(pr.h, W, draft, pr.u_accept, pr.u_resample,
                                                                mode=mode, out=out, workspace=ws),
                            args.sweep_steps, flush)
            check_device_error()
            outs[mode] = out
            logit = {"plain": 8 * rows * VOCAB, "stats_store": 4 * rows * VOCAB + 8 * 2 * b * VOCAB,
                     "stats_recompute": 8 * 2 * b * VOCAB}[mode]
            res.append({"batch": b, "mode": mode, "ms": round(ms, 4),
                        "tflops": round(flops / (ms / 1e3) / 1e12, 1),
                        "frac_of_bf16_peak": round(flops / (ms / 1e3) / 1e12 / tflops, 4),
                        "logit_bytes": logit,
                        "tokens_per_s": round(int(out[2].sum()) / (ms / 1e3), 1)})
            del ws
        same = all(all(torch.equal(x, y) for x, y in zip(outs["plain"], outs[m])) for m in outs)
        for e in res[-3:]:
            e["same_outputs_as_plain"] = same
        del pr, W, draft, outs
        torch.cuda.empty_cache()
    return res


def tree_sweep(args, dev, hbm):
    """The tree sampler's verification on top-k trees (children of each node =
    its most likely tokens, so acceptance is realistic) at vocab 128256: node
    rows read once (4 bytes per logit) plus one race row."""
    import torch
    from lossless_draft_verify_gated_b300 import binding, inputs
    flush = make_flusher(dev, args.l2_flush)
    res = []
    for b, widths in SWEEP_TREE:
        n1 = 1
        level = 1
        for w in widths:
            level *= w
            n1 += level
        lg = inputs.normal((b, n1, VOCAB), 8.0, f"tree.lg.B{b}.N{n1}", device=dev)
        par = torch.full((b, n1), -1, dtype=torch.int32, device=dev)
        tok = torch.zeros((b, n1), dtype=torch.int32, device=dev)
        # top-k children, breadth first (the drafting half of the tree sampler)
        nxt, frontier = 1, [0]
        for w in widths:
            new = []
            for node in frontier:
                top = torch.topk(lg[:, node], w, dim=-1).indices.to(torch.int32)
                for k in range(w):
                    par[:, nxt] = node
                    tok[:, nxt] = top[:, k]
                    new.append(nxt)
                    nxt += 1
            frontier = new
        ua = inputs.uniform_accept((b, n1), f"tree.ua.B{b}", device=dev)
        ur = inputs.uniform_race((b, VOCAB), f"tree.ur.B{b}", device=dev)
        ws = torch.empty(binding.uno_tree_verify_workspace(b, n1 - 1, VOCAB), dtype=torch.uint8, device=dev)
        out = (torch.empty(b, dtype=torch.int32, device=dev), torch.empty((b, n1 - 1), dtype=torch.int32, device=dev),
               torch.empty((b, n1), dtype=torch.int32, device=dev), torch.empty(b, dtype=torch.int32, device=dev),
               torch.empty(b, dtype=torch.int32, device=dev))
        ms = time_graph(lambda: binding.uno_tree_verify(lg, par, tok, ua, ur, out=out, workspace=ws),
                        args.sweep_steps, flush)
        by = 4 * b * n1 * VOCAB + 8 * b * VOCAB
        res.append({"batch": b, "nodes": n1, "widths": list(widths), "ms": round(ms, 5),
                    "mean_accepted_depth": round(float(out[0].float().mean()), 3),
                    "tokens_per_s": round(int(out[3].sum()) / (ms / 1e3), 1),
                    "bytes": by, "frac_hbm": round(by / (ms / 1e3) / 1e9 / hbm, 4)})
        del lg, ws
        torch.cuda.empty_cache()
    return res


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
        tm = Timer(st, dev, graph=not args.no_graph, l2_flush=args.l2_flush)
        tm.warm(args.warmup)
        check_device_error()
        barrier = torch.distributed.barrier if ws > 1 else None
        t_step, t_proj, t_ver, wall = tm.run(K, barrier)
    device_error = check_device_error()
    res, tokens_run = st.verify_results(K)
    assert all(int(r[3].abs().sum()) == 0 for r in res)
    # tokens per step of this replica, summed over the replicas
    ms_step, tokens_all = aggregate(sum(t_step) / K, tokens_run / K, ws, dev)
    tokens = tokens_all / ws  # per replica (every replica runs the same seeded steps)
    value = tokens_all / (ms_step / 1e3)

    # roofline of the dominant op: the layer's gated-LoRA projections
    ms_proj = statistics.mean(t_proj)
    ms_ver = statistics.mean(t_ver)
    bound, achieved, peak, unit, by, fl = proj_roofline(st.M, st.n_gate1, ms_proj, hbm, tflops)
    n_race = statistics.mean(int((r[0] < BLOCK).sum()) for r in res)
    vb = verify_bytes(args.batch, n_race, args.resample)
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_dict(args, args.batch, ws),
        "verified_tokens_per_step": round(tokens, 3),
        "verifier_input_sets": len(st.vsets),
        "launch": ("one CUDA graph per step; projections and verifier also timed alone, a graph each, "
                   "for their fields" if tm.g_step else
                   "CUDA graph per half-step" if tm.g_ver is not None else "eager"),
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
        out["e2e"] = e2e(st, dev, e2e_steps(K, len(st.vsets)), ws)
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


def e2e_steps(K, n_sets):
    """Steps of the end-to-end figure: the verifier input sets of the K
    device-timed steps, all K of them when they are at most one round of the
    n sets, else whole rounds (the mean that many rounds approach), about 50
    steps where a round is shorter."""
    return K if K <= n_sets else n_sets * max(1, min(K, 50) // n_sets)


def e2e(st, dev, steps, ws=1):
    """Same metric through the public API with host buffers: every step copies
    its inputs host->device from pinned memory, runs the ops eagerly and reads
    the verified tokens back.  Step i verifies input set i mod n, as the
    device-timed steps do.  The copies run on two copy streams, as a serving
    loop would issue them: a set's inputs as soon as its buffers' previous step
    has verified them, the layer's inputs once the previous step's projections
    have read theirs.  Also reported: the time of the copies alone and the host
    time spent in the API calls (enqueue, no synchronisation)."""
    import torch
    layer_host = []
    seen = set()
    for _, p in st.layer:
        for t in (p.x, p.gate):
            if t.data_ptr() not in seen:  # q/k/v and gate/up share their input; one gate tensor
                seen.add(t.data_ptr())
                layer_host.append((t.cpu().pin_memory(), t))
    n = min(steps, len(st.vsets))
    set_host = [[(st.vsets[k][f].cpu().pin_memory(), st.vsets[k][f]) for f in ("p", "q", "draft", "ua", "ur")]
                for k in range(n)]
    h2d = sum(h.numel() * h.element_size() for h, _ in layer_host + set_host[0])
    outs = [[torch.empty_like(st.vsets[k]["vout"][i], device="cpu").pin_memory() for i in (1, 2)]
            for k in range(n)]
    d2h = sum(o.numel() * o.element_size() for o in outs[0])
    torch.cuda.synchronize()

    def copies(k):
        for h, d in layer_host + set_host[k]:
            d.copy_(h, non_blocking=True)

    main = torch.cuda.current_stream()
    s_layer, s_set = torch.cuda.Stream(), torch.cuda.Stream()
    x_read = torch.cuda.Event()                         # the last step's projections are done
    set_free = [torch.cuda.Event() for _ in range(n)]   # set k's last verification is done
    x_in, set_in = torch.cuda.Event(), torch.cuda.Event()

    def start():
        # nothing of the pipeline starts before this point of the main stream
        ev = torch.cuda.Event()
        ev.record(main)
        s_layer.wait_event(ev)
        s_set.wait_event(ev)

    def one(i):
        k = i % n
        with torch.cuda.stream(s_set):
            if i >= n:
                s_set.wait_event(set_free[k])
            for h, d in set_host[k]:
                d.copy_(h, non_blocking=True)
            set_in.record(s_set)
        with torch.cuda.stream(s_layer):
            if i > 0:
                s_layer.wait_event(x_read)
            for h, d in layer_host:
                d.copy_(h, non_blocking=True)
            x_in.record(s_layer)
        main.wait_event(x_in)
        st.projections()
        x_read.record(main)
        main.wait_event(set_in)
        st.verify(k)
        set_free[k].record(main)
        outs[k][0].copy_(st.vsets[k]["vout"][1], non_blocking=True)
        outs[k][1].copy_(st.vsets[k]["vout"][2], non_blocking=True)

    start()
    for i in range(3):
        one(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # the copies alone
    e0.record()
    for i in range(steps):
        copies(i % n)
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
    start()
    for i in range(steps):
        one(i)
    e1.record()
    torch.cuda.synchronize()
    check_device_error()
    # every set's outputs are the same at each of its steps (seeded inputs)
    per_step = sum(int(outs[i % n][1].sum()) for i in range(steps)) / steps
    ms, tokens = aggregate(e0.elapsed_time(e1) / steps, per_step, ws, dev)
    return {"value": round(tokens / (ms / 1e3), 2), "unit": UNIT, "ms_per_step": round(ms, 4),
            "steps": steps, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "h2d_ms_per_step": round(ms_copy, 4), "host_api_ms_per_step": round(t_api / steps * 1e3, 4),
            "launch": "eager API calls; the host-to-device copies on two copy streams, overlapping "
                      "the previous step's kernels"}


def cpu_verify_set(batch, sigma, k):
    """Verifier input set k drawn on the host (CPU generators, as the GPU arm
    draws it for the headline), drafts drawn by the oracle's own sampler."""
    from lossless_draft_verify_gated_b300 import inputs
    import oracle
    vp = inputs.verify_problem(batch, BLOCK, VOCAB, sigma=sigma, seed=inputs.BASE_SEED + k)
    draft, _, margin = oracle.draft_sample(vp.q_logits, vp.u_draft)
    return vp, draft.reshape(batch, BLOCK), margin.reshape(batch, BLOCK)


def cpu_inputs(batch, sigma):
    """The same workload drawn on the host (CPU generators): the layer and
    verifier input set 0."""
    from lossless_draft_verify_gated_b300 import inputs
    M = 2 * BLOCK * batch
    layer = inputs.llama3_layer(M, rank=RANK, alpha=ALPHA, block=BLOCK)
    return (layer,) + cpu_verify_set(batch, sigma, 0)


class OracleStep:
    """The fp64 oracle as it stands, run on a bounded sample of one step and
    scaled to a full step.  Rows and output columns of a projection are
    independent, and so are sequences of the verifier, so the time of the
    sample scales by (rows x columns) and by sequences."""

    def __init__(self, batch, sigma):
        import oracle
        oracle.build()
        self.batch, self.sigma = batch, sigma
        self.M = 2 * BLOCK * batch
        self.layer, self.vp, self.draft, self.draft_margin = cpu_inputs(batch, sigma)
        self.nsets = n_verify_sets(batch)
        self.vsets = {0: (self.vp, self.draft, self.draft_margin)}
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

    def vset(self, k):
        """Verifier input set k (drawn on first use, outside any timing)."""
        if k not in self.vsets:
            self.vsets[k] = cpu_verify_set(self.batch, self.sigma, k)
        return self.vsets[k]

    def verify_sample(self, k):
        """The oracle's verifier on the sampled sequences of set k."""
        import oracle
        vp, draft, _ = self.vset(k)
        s = self.seqs
        return oracle.verify_block(vp.p_logits[:s], vp.q_logits[:s], draft[:s], vp.u_accept[:s],
                                   vp.u_resample[:s])

    def mean_tokens(self):
        """Verified tokens per step averaged over the sets that consecutive steps
        cycle through (the sampled sequences of each, scaled to the batch)."""
        return sum(float(self.verify_sample(k).n_emitted.sum()) for k in range(self.nsets)) \
            * (self.batch / self.seqs) / self.nsets

    def run(self, k=0):
        """One timed sample of the step, its verifier on input set k."""
        import oracle
        self.vset(k)
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
            r = self.verify_sample(k)
            t2 = time.perf_counter()
            tp += t1 - t0
            tv += t2 - t1
        self.last = (r_idx, ys, r) if k == 0 else None
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
    t_full, _, t_cpu = ob.run()
    # tokens per step: the mean over the verifier input sets that the GPU arm's
    # steps cycle through (the oracle's verifier on each set's sampled sequences)
    tokens = ob.mean_tokens()
    out = {"value": round(tokens / t_full, 4), "unit": UNIT, "cores": ob.threads, "kind": "oracle",
           "sample": ob.describe(1) + f"; {t_cpu:.1f} s of CPU work; verified tokens per step: the "
                     f"oracle's mean over the {ob.nsets} verifier input set(s) of the step",
           "verified_tokens_per_step": round(tokens, 3),
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
        # timed step j verifies input set j mod n, as the GPU arm's step j does
        j = i - args.warmup if i >= args.warmup else i
        t_full, tokens, _ = ob.run(j % ob.nsets)
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
                         "sample": ob.describe(args.steps) +
                                   f"; timed step j verifies input set j mod {ob.nsets}"},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }), flush=True)


def run_profile(args):
    """A few replays of one op for ncu: its launches are those of the sweep's
    figure for the same batch (and, for the LM head, strategy)."""
    import torch
    from lossless_draft_verify_gated_b300 import binding, inputs
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    b = args.batch
    if args.profile == "lm_head":
        pr = inputs.lm_head_problem(b, BLOCK, VOCAB, LM_D, device=dev)
        draft = torch.randint(0, VOCAB, (b, BLOCK), dtype=torch.int32, device=dev,
                              generator=inputs.generator("profile.draft", device=dev))
        ws = torch.empty(binding.uno_lm_head_verify_workspace(b, BLOCK, BLOCK, VOCAB, LM_D, args.lm_mode),
                         dtype=torch.uint8, device=dev)
        fn = lambda: binding.uno_lm_head_verify(pr.h, pr.W, draft, pr.u_accept, pr.u_resample,  # noqa: E731
                                                mode=args.lm_mode, workspace=ws)
    else:
        widths, n1, level = (3, 2, 2, 1), 1, 1
        for w in widths:
            level *= w
            n1 += level
        lg = inputs.normal((b, n1, VOCAB), 8.0, f"tree.lg.B{b}.N{n1}", device=dev)
        par = torch.full((b, n1), -1, dtype=torch.int32, device=dev)
        tok = torch.zeros((b, n1), dtype=torch.int32, device=dev)
        par[:, 1:] = 0  # a star of n1-1 children at the root: the widest walk
        tok[:, 1:] = torch.topk(lg[:, 0], n1 - 1, dim=-1).indices.to(torch.int32)
        ua = inputs.uniform_accept((b, n1), f"tree.ua.B{b}", device=dev)
        ur = inputs.uniform_race((b, VOCAB), f"tree.ur.B{b}", device=dev)
        fn = lambda: binding.uno_tree_verify(lg, par, tok, ua, ur)  # noqa: E731
    flush = make_flusher(dev, args.l2_flush)
    for _ in range(args.warmup + args.steps):
        flush()
        fn()
    torch.cuda.synchronize()
    check_device_error()


def main():
    args = parse()
    if args.profile:
        run_profile(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_uno(args)


if __name__ == "__main__":
    main()
