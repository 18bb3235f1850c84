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
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--sigma", type=float, default=SIGMA)
    ap.add_argument("--impl", choices=["uno", "reference"], default="uno")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
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
    """nvidia-smi sampling of SM clocks and throttle reasons during a run."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
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


class Step:
    """All inputs, outputs and workspaces of one step, resident on the device."""

    def __init__(self, batch, sigma, device, grouping="layer", temperature=1.0, resample="race"):
        import torch
        from lossless_draft_verify_gated_b300 import binding, inputs
        self.batch, self.device = batch, device
        self.M = 2 * BLOCK * batch
        self.layer = inputs.llama3_layer(self.M, rank=RANK, alpha=ALPHA, block=BLOCK, device=device)
        by_name = dict(self.layer)
        self.ys = {n: torch.empty((self.M, p.W.shape[0]), dtype=torch.bfloat16, device=device)
                   for n, p in self.layer}
        self.groups = []
        for names in GROUPINGS[grouping]:
            probs = [(by_name[n].x, by_name[n].W, by_name[n].A, by_name[n].B, by_name[n].gate,
                      by_name[n].alpha, self.ys[n]) for n in names]
            shapes = [(p[0].shape[1], p[1].shape[0], p[2].shape[0]) for p in probs]
            ws = torch.empty(binding.uno_gated_lora_linear_batched_workspace(shapes, self.M, 1),
                             dtype=torch.uint8, device=device)
            self.groups.append((probs, ws))
        vp = inputs.verify_problem(batch, BLOCK, VOCAB, sigma=sigma, device=device)
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
        self.n_gate1 = int(self.layer[0][1].gate.sum())
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


def run_uno(args):
    import torch
    ws, rank, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    from lossless_draft_verify_gated_b300 import binding
    binding.lib()
    hbm, tflops, tflops_sustained, peak_kind = peaks()
    st = Step(args.batch, args.sigma, dev, args.grouping, args.temperature, args.resample)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)

    # CUDA graphs of the two halves of the step (launch overhead off the clock)
    g_proj = g_ver = None
    if not args.no_graph:
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            st.projections()
            st.verify()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g_proj, g_ver = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_proj):
            st.projections()
        with torch.cuda.graph(g_ver):
            st.verify()

    def run_proj():
        g_proj.replay() if g_proj is not None else st.projections()

    def run_ver():
        g_ver.replay() if g_ver is not None else st.verify()

    for _ in range(args.warmup):
        flush.zero_()
        run_proj()
        run_ver()
    torch.cuda.synchronize()
    assert binding.uno_device_error() == 0

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    with Clocks(local) as clk:
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(K):
            flush.zero_()  # L2 flush, outside the timed events
            ev[i][0].record()
            run_proj()
            ev[i][1].record()
            run_ver()
            ev[i][2].record()
        torch.cuda.synchronize()
        if ws > 1:
            torch.distributed.barrier()
        wall = time.perf_counter() - t0
    t_step = [e[0].elapsed_time(e[2]) for e in ev]
    t_proj = [e[0].elapsed_time(e[1]) for e in ev]
    t_ver = [e[1].elapsed_time(e[2]) for e in ev]
    n_acc, toks, n_em, vstat = (t.cpu() for t in st.vout)
    assert int(vstat.abs().sum()) == 0
    ms_step, tokens_all = aggregate(sum(t_step) / K, int(n_em.sum()), ws, dev)
    tokens = tokens_all // ws  # per replica (every replica runs the same seeded step)
    value = tokens_all / (ms_step / 1e3)

    # roofline of the dominant op: the layer's gated-LoRA projections
    by, fl = proj_bytes_flops(st.M, st.n_gate1)
    ms_proj = statistics.mean(t_proj)
    ms_ver = statistics.mean(t_ver)
    ai = fl / by
    bound = "hbm" if ai < (tflops * 1e12) / (hbm * 1e9) else "tensor"
    if bound == "hbm":
        achieved, peak, unit = by / (ms_proj / 1e3) / 1e9, hbm, "GB/s"
    else:
        achieved, peak, unit = fl / (ms_proj / 1e3) / 1e12, tflops, "TFLOP/s"
    n_race = int((n_acc < BLOCK).sum())
    vb = verify_bytes(args.batch, n_race, args.resample)
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_name(args.batch), "batch": args.batch, "block": BLOCK,
                   "vocab": VOCAB, "rank": RANK, "alpha": ALPHA, "sigma": args.sigma,
                   "rows_per_projection": st.M, "verified_tokens_per_step": tokens,
                   "l2": "flushed before every step (2x L2 write, outside the timed events)",
                   "launch": "CUDA graph per half-step" if g_proj is not None else "eager",
                   "grouping": args.grouping + ": " + " | ".join(",".join(g) for g in GROUPINGS[args.grouping]),
                   "sampler": f"temperature {args.temperature}, {args.resample} resample",
                   "parallelism": f"dp{ws} (independent replicas, no collective)"},
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
            out["cpu_baseline"] = cpu_baseline(st, args.batch, args.sigma, budget_s=15.0)
        else:  # the timed oracle step is the default sampler's
            out["cpu_baseline"] = None
    if rank == 0:
        print(json.dumps(out), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def e2e(st, dev, steps, ws=1):
    """Same metric through the public API with host buffers: every step copies
    its inputs host->device from pinned memory, runs the ops eagerly and reads
    the verified tokens back."""
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

    def one():
        for h, d in host.values():
            d.copy_(h, non_blocking=True)
        st.projections()
        st.verify()
        outs[0].copy_(st.vout[1], non_blocking=True)
        outs[1].copy_(st.vout[2], non_blocking=True)

    for _ in range(3):
        one()
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        one()
    e1.record()
    torch.cuda.synchronize()
    ms, tokens = aggregate(e0.elapsed_time(e1) / steps, int(outs[1].sum()), ws, dev)
    return {"value": round(tokens / (ms / 1e3), 2), "unit": UNIT, "ms_per_step": round(ms, 4),
            "steps": steps, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "launch": "eager API calls"}


def cpu_inputs(batch, sigma):
    """The same workload generated on the host (CPU generators), drafts drawn
    by the oracle's own sampler."""
    from lossless_draft_verify_gated_b300 import inputs
    import oracle
    M = 2 * BLOCK * batch
    layer = inputs.llama3_layer(M, rank=RANK, alpha=ALPHA, block=BLOCK)
    vp = inputs.verify_problem(batch, BLOCK, VOCAB, sigma=sigma)
    draft, _, _ = oracle.draft_sample(vp.q_logits, vp.u_draft)
    return layer, vp, draft.reshape(batch, BLOCK)


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
        self.layer, self.vp, self.draft = cpu_inputs(batch, sigma)
        self.threads = oracle.num_threads()
        self.rows = min(self.M, max(2, self.threads))
        self.seqs = min(batch, max(1, self.threads))
        self.col_frac = 1.0
        self.repeat = 1  # samples per timed step (a small step is repeated to time it reliably)

    def run(self):
        import numpy as np
        import oracle
        M, rows = self.M, self.rows
        r_idx = np.concatenate([np.arange(rows // 2), M - 1 - np.arange(rows - rows // 2)])
        tp = tv = 0.0
        for _ in range(self.repeat):
            t0 = time.perf_counter()
            scale_p = 0.0
            for _, p in self.layer:
                d_out = p.W.shape[0]
                c = max(8, int(round(d_out * self.col_frac / 8)) * 8)
                c = min(c, d_out)
                oracle.gated_lora_linear(p.x[r_idx], p.W[:c], p.A, p.B[:c], p.gate[r_idx], p.alpha)
                scale_p = (M / rows) * (d_out / c)  # equal fractions for every projection
            t1 = time.perf_counter()
            s = self.seqs
            vp = self.vp
            r = oracle.verify_block(vp.p_logits[:s], vp.q_logits[:s], self.draft[:s], vp.u_accept[:s],
                                    vp.u_resample[:s])
            t2 = time.perf_counter()
            tp += t1 - t0
            tv += t2 - t1
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


def cpu_baseline(st, batch, sigma, budget_s=15.0):
    ob = OracleStep(batch, sigma)
    ob.calibrate(budget_s)
    t_full, tokens, t_cpu = ob.run()
    return {"value": round(tokens / t_full, 4), "unit": UNIT, "cores": ob.threads, "kind": "oracle",
            "sample": ob.describe(1) + f"; {t_cpu:.1f} s of CPU work",
            "ms_per_step_extrapolated": round(t_full * 1e3, 2)}


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
        "config": {"workload": workload_name(args.batch), "batch": args.batch, "block": BLOCK,
                   "vocab": VOCAB, "rank": RANK, "alpha": ALPHA, "sigma": args.sigma},
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
