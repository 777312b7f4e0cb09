"""Decode-step benchmark: tokens/s and achieved HBM GB/s of the GB300 step.

One "step" = one dec_step call (the whole decode path: embedding, every layer,
lm_head and argmax) for one batch, followed by the greedy feedback kernel
(token <- argmax, position += 1).  Inputs are seeded synthetic tensors already
resident in HBM; the per-step weights (> 1 GB for every model-sized workload)
are larger than L2, so no flush is needed between steps.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--repeats R] [--config NAME]
                       [--impl ours|reference] [--no-cpu-baseline]
The default workload is qwen3-8b-b1, the batch-1 Qwen3-8B-shaped bf16 step; the timed
region is R (default 5) repeats of K steps from the same starting tokens and positions,
and the line reports the median repeat.
With --gpus N > 1 (launched by torchrun) every rank runs an independent replica
of the workload on its own GPU (the step has no cross-sequence exchange); the
value is the sum of all ranks' tokens over the slowest rank's time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import pathlib
import statistics
import subprocess
import sys
import threading
import time

ROOT = pathlib.Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

DEFAULT_CONFIG = "qwen3-8b-b1"  # the batch-1 Qwen3-8B-shaped bf16 step (the >= 70% of peak HBM target)
METRIC = "decode tokens/s and achieved HBM GB/s (fraction of GB300 peak) per step"

# ncu DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch of the
# dominant kernel class, keyed by workload and class, valid only for the kernel
# sources whose digest is recorded with it (see profiles/).  "alg": the captured launch's
# algorithmic bytes where the capture's cached lengths differ from the bench's (attention):
# the traffic is then scaled to the bench launch (it grows with the positions read).
# Captured with token_decode_step_gb300.profile_case (2 layers, same shapes as the bench
# workload) under `ncu --set full`; profiles/ holds the summaries and commands.
NCU_TRAFFIC: dict = {
    "qwen3-0.6b": {"attention": {"bytes": 4263680, "alg": 4203008, "src": "attention", "csrc": "7606bcbf82634d56"}},
    "qwen3-8b-b1": {"gate_up": {"bytes": 201391360 + 3057152, "src": "gemv", "csrc": "9b1e690fbc265ef7"}},
    "qwen3-8b-b1-kv8": {"gate_up": {"bytes": 201391360 + 3057152, "src": "gemv", "csrc": "9b1e690fbc265ef7"}},
    "qwen3-4b-q4": {"gate_up": {"bytes": 28072448, "src": "gemv", "csrc": "9b1e690fbc265ef7"}},
    "qwen3-8b-b8": {"gate_up": {"bytes": 201520128 + 2948096, "src": "gemm_tc", "csrc": "560790667e6b9504",
                                "proj": [0, 1]}},
    "qwen3-8b-q4-b32": {"attention": {"bytes": 607751680 + 4087552, "alg": 606966272, "src": "attention",
                                      "csrc": "7606bcbf82634d56"}},
    "qwen3-8b-q4-b32-kv8": {"attention": {"bytes": 299072512 + 3900672, "alg": 298216720, "src": "attention",
                                          "csrc": "7606bcbf82634d56"}},
}


# the sources each captured kernel is built from (a recorded traffic stays valid while they
# are unchanged)
KERNEL_SOURCES = {
    "attention": ["k_attention.cu", "k_attention_q8.cu", "attn_common.cuh"],
    "gemv": ["k_gemv1.cu", "gemv_common.cuh", "q4.cuh"],
    "gemm_tc": ["k_gemm_tc.cu", "q4.cuh"],
}


def csrc_digest(files=None) -> str:
    h = hashlib.sha256()
    csrc = ROOT / "token_decode_step_gb300" / "csrc"
    paths = sorted(csrc.glob("*.cu*")) if files is None else [csrc / f for f in sorted(files)]
    for p in paths:
        h.update(p.read_bytes())
    return h.hexdigest()[:16]


def measured_peaks() -> tuple[dict, str]:
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        return json.loads(p.read_text()), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


class ClockSampler:
    """nvidia-smi SM clock / throttle sampling around the timed region.

    Sampling starts (and its first sample is awaited) before the timed region;
    begin() and end() mark the region on the host clock and summary() keeps the
    samples stamped inside it.  If the region is shorter than one sampling period,
    the first sample after begin() stands in and `samples_in_region` says so.
    """

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 20

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[tuple[float, str]] = []
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.PERIOD_MS)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            deadline = time.time() + 3.0
            while not self.lines and time.time() < deadline:
                time.sleep(0.01)
        except FileNotFoundError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def begin(self):
        self.t0 = time.time()

    def end(self):
        self.t1 = time.time()
        # one more period so that a sample stamped inside the region has been read
        time.sleep(2 * self.PERIOD_MS / 1000.0)

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    @staticmethod
    def _stamp(text: str) -> float | None:
        import datetime
        try:
            return datetime.datetime.strptime(text.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def summary(self) -> dict:
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        for arrival, ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            t = self._stamp(parts[0])
            rows.append((t if t is not None else arrival, parts[1:]))
        inside = [r for r in rows if self.t0 is not None and self.t1 is not None and self.t0 <= r[0] <= self.t1]
        n_in = len(inside)
        if not inside and self.t0 is not None:
            after = [r for r in rows if r[0] >= self.t0]
            inside = after[:1]
        sm, smax, reasons = [], None, set()
        for _, parts in inside:
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm), "samples_in_region": n_in}


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time: every rank contributes its own, all receive the maximum
    (replicas run independently; the job is done when the last one is)."""
    if world <= 1:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, batch: int, steps: int, ms_max: float) -> float:
    """Whole-job throughput: the tokens of every rank over the slowest rank's time."""
    return world * batch * steps / (ms_max / 1e3)


def run_ours(args, rank: int, world: int) -> dict | None:
    import numpy as np
    import torch
    import synthetic
    from token_decode_step_gb300 import build as build_mod
    if rank == 0 or not (ROOT / "token_decode_step_gb300" / "libdec.so").exists():
        build_mod.build()
    if world > 1:
        torch.distributed.barrier()
    from token_decode_step_gb300 import dec as D
    from token_decode_step_gb300.torch_glue import Decoder

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    wl0 = synthetic.WORKLOADS[args.config]
    total = args.warmup + args.steps + args.profile_steps + args.e2e_steps + 2  # the repeats rewind
    wl = wl0.replace(steps=total)  # cache capacity for every step this run takes
    model = synthetic.generate(wl, device=dev)
    dec = Decoder(wl, model, proj_kernels=args.proj)
    B, V = wl.batch, wl.vocab
    tokens = model["tokens"].clone()
    positions = model["positions"].clone()
    kv = synthetic.kv_buffer(model["kv"])  # the one flat cache buffer the library reads
    logits = torch.empty((B, V), dtype=torch.float32, device=dev)
    argmax = torch.empty((B,), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    p0 = float(model["positions"].float().mean())

    def one_step():
        dec.step(tokens, positions, kv, logits, argmax, stream)
        dec.advance(argmax, tokens, positions, stream)

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize(dev)
    pos_start = float(positions.float().mean())
    # every repeat starts from the same tokens and positions (the cache slots it writes are
    # rewritten), so the repeats time the same work; the line reports the median repeat
    tok0, pos0 = tokens.clone(), positions.clone()
    rep_ms = []
    with ClockSampler(dev.index) as clk:
        for rep in range(args.repeats):
            tokens.copy_(tok0)
            positions.copy_(pos0)
            if world > 1:
                torch.distributed.barrier()
            torch.cuda.synchronize(dev)
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            if rep == 0:
                clk.begin()
            ev0.record(stream)
            for _ in range(args.steps):
                one_step()
            ev1.record(stream)
            torch.cuda.synchronize(dev)
            if world > 1:
                torch.distributed.barrier()
            rep_ms.append(max_over_ranks(ev0.elapsed_time(ev1), world, dev))
        clk.end()
    ms = statistics.median(rep_ms)
    mean_p = pos_start + (args.steps - 1) / 2.0  # mean cached length over the timed steps

    # per-kernel-class durations: the same step with per-launch CUDA events (no graph)
    cls_ms = [0.0] * D.DEC_K_COUNT
    cls_n = [0] * D.DEC_K_COUNT
    prof_p = float(positions.float().mean())
    for _ in range(args.profile_steps):
        dec.profile_step(tokens, positions, kv, logits, argmax, cls_ms, cls_n, stream)
        dec.advance(argmax, tokens, positions, stream)
    torch.cuda.synchronize(dev)
    prof_mean_p = prof_p + (args.profile_steps - 1) / 2.0

    # end to end through the C ABI with host buffers (dec_step_host): the host greedy loop's
    # call, H2D of tokens + positions, the step and D2H of the argmax inside it, every step
    h_tok = tokens.cpu().numpy().astype(np.int32).copy()
    h_pos = positions.cpu().numpy().astype(np.int32).copy()
    def e2e_step():
        dec.step_host(h_tok, h_pos, kv, None, h_tok, stream)  # the argmax overwrites the tokens
        h_pos[...] += 1

    e2e_step()  # captures the graph for this pointer set (untimed)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        e2e_step()
    e2e_s = time.perf_counter() - t0

    # the sampling kernel (dec_sample, the step after the argmax) on this step's logits;
    # a separate entry point, not part of the timed step
    prm = D.SamplingParams(temperature=0.8, top_k=50, top_p=0.9, seed=1, offset=0, offset_device=None)
    stok = torch.empty((B,), dtype=torch.int32, device=dev)
    for _ in range(3):
        D.dec_sample(logits.data_ptr(), B, V, prm, stok.data_ptr(), stream.cuda_stream)
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_samp = 20
    s0.record(stream)
    for i in range(n_samp):
        prm.offset = i
        D.dec_sample(logits.data_ptr(), B, V, prm, stok.data_ptr(), stream.cuda_stream)
    s1.record(stream)
    torch.cuda.synchronize(dev)
    samp_us = s0.elapsed_time(s1) * 1000.0 / n_samp
    sampling = {"us_per_call": round(samp_us, 2), "rows": B, "vocab": V,
                "params": "temperature 0.8, top_k 50, top_p 0.9", "logit_bytes": B * V * 4,
                "logit_gbs": round(B * V * 4 / (samp_us * 1e-6) / 1e9, 1)}

    # optional: a multi-token step (tokens_per_seq T: a verify step, or a prefill chunk
    # of T prompt tokens per sequence) on the same weights and cache, one graph replay per
    # step, same tokens and positions every time (the K/V slots are rewritten with the
    # same values); its logits are not written (a prefill keeps only the cache)
    def multi_token(T: int, n: int) -> tuple[float, dict]:
        vdec = Decoder(wl, model, tokens_per_seq=T, proj_kernels=args.proj)
        vt = torch.randint(0, V, (B * T,), dtype=torch.int32, device=dev)
        va = torch.empty((B * T,), dtype=torch.int32, device=dev)
        vpos = torch.zeros_like(positions) if T > 8 else positions.clone()
        for _ in range(3):
            vdec.step(vt, vpos, kv, None, va, stream)
        v0, v1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        v0.record(stream)
        for _ in range(n):
            vdec.step(vt, vpos, kv, None, va, stream)
        v1.record(stream)
        torch.cuda.synchronize(dev)
        # the same step with per-launch events: milliseconds per kernel class (attention
        # includes the K/V append pass)
        pm, pn = [0.0] * D.DEC_K_COUNT, [0] * D.DEC_K_COUNT
        vdec.profile_step(vt, vpos, kv, None, va, pm, pn, stream)
        torch.cuda.synchronize(dev)
        vdec.close()
        tot = sum(pm)
        by_class = {name: {"ms": round(pm[c], 4), "share": round(pm[c] / tot, 4) if tot > 0 else None}
                    for c, name in enumerate(D.KERNEL_CLASS_NAMES)}
        return v0.elapsed_time(v1) / n, by_class

    verify = None
    if args.verify > 1:
        T = args.verify
        vms, vcls = multi_token(T, 20)
        verify = {"kernel_classes": vcls, "tokens_per_seq": T, "rows": B * T, "ms_per_verify": round(vms, 4),
                  "one_token_ms": round(ms / args.steps, 4), "verify_over_one": round(vms / (ms / args.steps), 3),
                  "tokens_checked_per_s": round(B * T / (vms / 1e3), 1)}
    prefill = None
    if args.prefill > 1:
        T = args.prefill
        pms, pcls = multi_token(T, 5)
        prefill = {"kernel_classes": pcls, "tokens_per_seq": T, "rows": B * T, "positions": "0 .. T-1 of every sequence",
                   "ms_per_chunk": round(pms, 3), "prompt_tok_per_s": round(B * T / (pms / 1e3), 1)}

    per_step = [1, wl.n_layers, wl.n_layers, wl.n_layers, wl.n_layers, wl.n_layers, 1]  # launches per class
    bytes_step = sum(n * dec.kernel_bytes(c, mean_p) for c, n in enumerate(per_step))
    cls_bytes = [dec.kernel_bytes(c, prof_mean_p) for c in range(D.DEC_K_COUNT)]
    launches = dec.launches_per_step
    dec.close()
    return {"ms": ms, "rep_ms": rep_ms, "mean_p": mean_p, "bytes_step": bytes_step, "cls_ms": cls_ms, "cls_n": cls_n,
            "cls_bytes": cls_bytes, "e2e_s": e2e_s, "launches": launches, "wl": wl0, "B": B,
            "clocks": clk.summary(), "sampling": sampling, "verify": verify, "prefill": prefill}


def cpu_oracle_sample(config: str, warmup: int, steps: int, budget_s: float) -> dict:
    """Time the CPU oracle (as it stands) on whole greedy decode steps of the workload.

    A bounded sample: batched workloads run their first sequence only (its own KV
    cache and prompt token); `warmup` untimed steps (the first converts the weights
    to float64), then up to `steps` timed steps, stopping after the first one that
    ends past `budget_s`.
    """
    import numpy as np
    import oracle
    import synthetic
    import torch
    wl = synthetic.WORKLOADS[config].replace(steps=warmup + steps + 1)
    model = synthetic.generate(wl, device="cpu")
    m = oracle.OracleModel.from_synthetic(wl, model, cache_weights=True)
    bs = 1 if wl.batch > 1 else wl.batch
    if isinstance(model["kv"], dict):  # affine 8-bit cache
        kv = oracle.Affine8Cache(model["kv"]["codes"][:, :, :bs].contiguous().numpy().copy(),
                                 model["kv"]["params"][:, :, :bs].contiguous().view(torch.int16).numpy()
                                 .view(np.uint16).copy())
    else:
        kv = model["kv"][:, :, :bs].contiguous().view(torch.int16).numpy().view(np.uint16).copy()
    tokens = model["tokens"][:bs].numpy().copy()
    pos = model["positions"][:bs].numpy().copy()

    def step():
        nonlocal tokens, pos
        _, am = oracle.decode_step(m, kv, tokens, pos)
        tokens = am.astype(np.int32)
        pos = pos + 1

    for _ in range(warmup):
        step()
    done = 0
    t0 = time.perf_counter()
    while done < steps:
        step()
        done += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    seqs = f"sequence 0 of {wl.batch}" if bs < wl.batch else f"batch {wl.batch}"
    return {"value": bs * done / el, "unit": "tok/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} timed greedy step(s) of {config} ({seqs}) after {warmup} untimed "
                      f"(the first converts the weights to float64), {el:.1f} s"}


def workload_config(wl, world: int) -> dict:
    return {
        "workload": wl.name, "batch": wl.batch, "layers": wl.n_layers, "hidden": wl.hidden,
        "cached_positions": wl.prefill if not isinstance(wl.prefill, tuple) else list(wl.prefill),
        "weight_format": wl.weight_format, "kv_format": wl.kv_format, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        "l2": ("inputs larger than L2 (per-step weights exceed 129 MB); no flush" if weight_bytes(wl) > 129e6 else
               "inputs smaller than L2 and not flushed: a cache-warm number"),
    }


def weight_bytes(wl) -> float:
    """Bytes of every linear layer of the workload (bf16: 2 per weight, 4-bit: 0.5625)."""
    per = 2.0 if wl.weight_format == "bf16" else 0.5 + 4.0 / 64
    sh = wl.shapes()
    n = sum(a * b for k, (a, b) in sh.items() if k != "lm_head") * wl.n_layers + sh["lm_head"][0] * sh["lm_head"][1]
    return n * per


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=128)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--repeats", type=int, default=5, help="timed repeats of --steps steps; the median is reported")
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--profile-steps", type=int, default=8)
    ap.add_argument("--e2e-steps", type=int, default=32)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--proj", type=int, default=0, choices=[0, 1, 2],
                    help="dec_config.proj_kernels of the 2..32-row projections: 0 auto, 1 mma.sync, 2 tcgen05")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--verify", type=int, default=0,
                    help="also time the multi-token verify step with this many tokens per sequence (2..8)")
    ap.add_argument("--prefill", type=int, default=0,
                    help="also time one prefill chunk of T prompt tokens per sequence (tokens_per_seq = T)")
    ap.add_argument("--ref-budget", type=float, default=60.0,
                    help="reference arm: stop the timed oracle steps after this many seconds")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))

    if args.impl == "reference":
        # the reference arm is the CPU oracle, timed as it stands on the host cores (rank 0 only)
        if rank != 0:
            return
        import synthetic
        t0 = time.perf_counter()
        s = cpu_oracle_sample(args.config, args.warmup, args.steps, args.ref_budget)
        s["value"] = round(s["value"], 4)  # the line's value, once
        cfg = workload_config(synthetic.WORKLOADS[args.config], world)
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": s["value"], "unit": "tok/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1000.0 / s["value"], 2) if s["value"] else None, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded, random-init weights; see synthetic/workloads.py)",
            "config": cfg, "timing": "host wall clock over the timed oracle steps", "cpu_baseline": s,
            "e2e": {"value": s["value"], "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": round(time.perf_counter() - t0, 1),
        }))
        return

    import torch
    if world > 1:
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    r = run_ours(args, rank, world)
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return

    from token_decode_step_gb300 import dec as D
    wl, B = r["wl"], r["B"]
    peaks, peak_kind = measured_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    steps = args.steps
    tok_s = job_tokens_per_s(world, B, steps, r["ms"])
    step_ms = r["ms"] / steps
    step_gbs = r["bytes_step"] / (step_ms / 1e3) / 1e9

    # dominant kernel class by measured time
    cls_ms, cls_n = r["cls_ms"], r["cls_n"]
    dom = max(range(D.DEC_K_COUNT), key=lambda c: cls_ms[c])
    dom_name = D.KERNEL_CLASS_NAMES[dom]
    dom_avg_ms = cls_ms[dom] / max(1, cls_n[dom])
    line = {
        "metric": METRIC,
        "value": round(tok_s, 2),
        "unit": "tok/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if wl.weight_format == "bf16" else "int4-affine-g64",
        "data": "synthetic (seeded, random-init weights; see synthetic/workloads.py)",
        "config": workload_config(wl, world),
        "timing": (f"CUDA events on the launching stream, CUDA-graph replay per step; median of "
                   f"{len(r['rep_ms'])} repeats of {steps} steps"),
        "repeat_ms_per_step": [round(x / steps, 4) for x in r["rep_ms"]],
        "step_hbm_gbs": round(step_gbs, 1),
        "step_hbm_frac": round(step_gbs / hbm_peak, 4),
        "step_hbm_frac_of_nominal_8tbs": round(step_gbs / 8000.0, 4),
        "step_bytes": int(r["bytes_step"]),
        "peak_hbm_gbs": hbm_peak,
        "peak_kind": peak_kind,
        "gpu_launches": (r["launches"] + 1) * steps,
        "clocks": r["clocks"],
        "kernel_ms_per_launch": {D.KERNEL_CLASS_NAMES[c]: round(cls_ms[c] / max(1, cls_n[c]), 5)
                                 for c in range(D.DEC_K_COUNT)},
        "kernel_share": {D.KERNEL_CLASS_NAMES[c]: round(cls_ms[c] / max(1e-12, sum(cls_ms)), 4)
                         for c in range(D.DEC_K_COUNT)},
    }
    line["proj_kernels"] = {0: "auto", 1: "mma.sync", 2: "tcgen05"}[args.proj]
    line["sampling"] = r["sampling"]
    if r["verify"]:
        line["verify"] = r["verify"]
    if r["prefill"]:
        line["prefill"] = r["prefill"]
    e2e_tok_s = B * args.e2e_steps / r["e2e_s"]
    line["e2e"] = {"value": round(e2e_tok_s, 2), "unit": "tok/s", "h2d_bytes_per_step": 8 * B,
                   "d2h_bytes_per_step": 4 * B}
    db = r["cls_bytes"][dom]
    line["roofline"] = {"bound": "hbm", "kernel": dom_name, "achieved": None, "peak": hbm_peak, "unit": "GB/s",
                        "frac": None, "traffic": None}
    if db:
        ach = db / (dom_avg_ms / 1e3) / 1e9
        line["roofline"].update({"achieved": round(ach, 1), "frac": round(ach / hbm_peak, 4),
                                 "bytes_per_launch": int(db), "avg_launch_ms": round(dom_avg_ms, 5)})
        tr = NCU_TRAFFIC.get(args.config, {}).get(dom_name)
        if (tr and tr.get("src") in KERNEL_SOURCES and tr.get("csrc") == csrc_digest(KERNEL_SOURCES[tr["src"]])
                and args.proj in tr.get("proj", [0, 1, 2])):
            if tr.get("alg"):  # captured at other cached lengths: scaled to this launch's algorithmic bytes
                line["roofline"]["traffic"] = int(round(tr["bytes"] * db / tr["alg"]))
                line["roofline"]["traffic_note"] = (f"ncu capture of {tr['bytes']} bytes for {tr['alg']} algorithmic "
                                                    f"bytes, scaled to this launch")
            else:
                line["roofline"]["traffic"] = tr["bytes"]
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_sample(args.config, 1, 1000, args.cpu_budget)
    print(json.dumps(line))


if __name__ == "__main__":
    main()
