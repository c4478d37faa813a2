"""Benchmark: MSA training step (sparse forward + backward) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload msa_s64k_planted] [--no-cpu-baseline] [--no-e2e]
    python bench.py --workload msa_decode_b128     (decode step of inference; not the default)

One step = msa_forward (proxy top-k selection + sparse attention) followed by msa_backward
(dQ, dK, dV, dQp, dKp) on one batch of the workload, inputs resident in HBM.  Prints one JSON
line (rank 0).  N > 1 ranks (torchrun) each process their own batch: weak scaling, no data-path
collective; the time is the max over ranks.

--impl reference times the fp64 CPU oracle on the host cores over a bounded sample of the same
workload (tokens/s extrapolated from the sample), as the slow reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from block_sparse_attention_qp_gb300 import dist, flops  # noqa: E402
from block_sparse_attention_qp_gb300.inputs import WORKLOADS, make_inputs, workload_seed  # noqa: E402

METRIC = "MSA fwd+bwd tokens/s & TFLOP/s at 64K ctx; % of GB300 dense bf16 peak"
UNIT = "tokens/s"
L2_BYTES = 129 * 2 ** 20


def workload_by_name(name):
    for i, w in enumerate(WORKLOADS):
        if w.name == name:
            return i + 1, w
    raise SystemExit(f"unknown workload {name}; choose from {[w.name for w in WORKLOADS]}")


def input_bytes(w):
    """Bytes of the step's bf16 inputs q, k, v, qp, kp, dout."""
    return w.B * w.S * (2 * w.Hq + 2 * w.Hkv + w.Hp + 1) * w.D * 2


def config_of(w):
    inputs_bytes = input_bytes(w)
    return {"workload": w.name, "desc": w.describe(), "B": w.B, "S": w.S, "Hq": w.Hq,
            "Hkv": w.Hkv, "Hp": w.Hp, "d": w.D, "top_k": w.top_k, "block": 128,
            "planted_blocks": w.planted, "scale": w.scale,
            "l2": f"inputs larger than L2 ({inputs_bytes / 2**20:.0f} MiB > 129 MiB); no flush"}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "of measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "of fallback"


# ------------------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def _query(self, loop_ms=None):
        cmd = ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
               "--format=csv,noheader,nounits"]
        return cmd + (["-lms", str(loop_ms)] if loop_ms else [])

    @staticmethod
    def _parse(text):
        rows = []
        for line in text.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        return rows

    def __enter__(self):
        self.when = "during the timed region"
        try:
            self.proc = subprocess.Popen(self._query(50), stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            # the sampler is live once its first line is out (that line predates the region)
            self.proc.stdout.readline()
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.samples = []
        if self.proc is None:
            return False
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.samples = self._parse(out)
        if not self.samples:  # region shorter than one sampling interval: read once right after
            try:
                one = subprocess.run(self._query(), capture_output=True, text=True, timeout=10)
                self.samples = self._parse(one.stdout)
                self.when = "right after the timed region (shorter than one 50 ms sample)"
            except (OSError, subprocess.TimeoutExpired):
                pass
        return False

    def summary(self):
        if not getattr(self, "samples", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        mx = [float(s[2]) for s in self.samples if s[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in self.samples for i in range(4)
                          if s[5 + i].lower() == "active"})
        pw = [float(s[3]) for s in self.samples if s[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "power_w_max": max(pw) if pw else None, "samples": len(self.samples),
                "sampled": self.when}


# ------------------------------------------------------------------------------ oracle sample
def oracle_sample(w, x64, idx_rows_fn, tokens, threads=None):
    """Time the fp64 oracle on `tokens` (b, t) of workload w: their selection rows, their
    forward rows and their exact share of every gradient.  Returns seconds."""
    import oracle

    if threads:
        oracle.set_threads(threads)
    B, S = w.B, w.S
    t0 = time.perf_counter()
    rows = np.array([(b, g, t) for (b, t) in tokens for g in range(w.Hp)], np.int32)
    sel, _ = oracle.select(x64["qp"], x64["kp"], w.top_k, w.scale, rows=rows)
    idx = idx_rows_fn(rows, sel)
    frows = np.array([(b, t, h) for (b, t) in tokens for h in range(w.Hq)], np.int32)
    oracle.forward(x64["q"], x64["k"], x64["v"], idx, w.top_k, w.scale, rows=frows, Hp=w.Hp)
    mask = np.zeros((B, S), bool)
    for b, t in tokens:
        mask[b, t] = True
    oracle.backward(x64["q"], x64["k"], x64["v"], x64["qp"], x64["kp"], x64["dout"], idx,
                    w.top_k, w.scale, tok_mask=mask, only_masked=True)
    return time.perf_counter() - t0


def oracle_inputs(w, seed):
    import oracle

    x = make_inputs(w, seed)
    return {k: oracle.f64(v) for k, v in x.items() if isinstance(v, torch.Tensor)}


def idx_builder(w):
    """Sparse index map holding only the sampled rows (others -1: they are not visited)."""
    def build(rows, sel):
        idx = np.full((w.B, w.Hp, w.S, w.top_k), -1, np.int32)
        idx[rows[:, 0], rows[:, 1], rows[:, 2]] = sel
        return idx
    return build


def sample_tokens(w, n, rng):
    """Token positions spread over the sequence (the oracle's per-token cost grows with t)."""
    ts = rng.choice(w.S, size=n, replace=False)
    bs = rng.integers(0, w.B, size=n)
    return sorted(zip(bs.tolist(), ts.tolist()))


def run_reference(args, w, wi):
    world, rank, _ = dist.env_world()
    if rank != 0:
        return
    import oracle

    oracle.build()
    threads = oracle.threads()
    x64 = oracle_inputs(w, workload_seed(wi))
    rng = np.random.default_rng(0)
    n_tok = args.ref_tokens
    build = idx_builder(w)
    times = []
    for step in range(args.warmup + args.steps):
        toks = sample_tokens(w, n_tok, rng)
        dt = oracle_sample(w, x64, build, toks)
        if step >= args.warmup:
            times.append(dt)
    sec = sum(times) / len(times)
    value = n_tok / sec
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "cpu_model": cpu_model(),
                             "sample": f"{n_tok} random tokens per step (all {w.Hp} groups, "
                                       f"{w.Hq} heads): selection rows, forward rows and their "
                                       f"exact share of every gradient"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------ our arm
KERNEL_WORK = {
    # kernel name -> (bound, function(workload) -> algorithmic FLOPs per step; a kernel that runs
    # in passes over sequence chunks divides them over its launches)
    "proxy_topk": ("tensor", lambda w: 2 * w.D * flops.n_px(w.S) * w.Hp * w.B),
    "attn_fwd": ("tensor", lambda w: 4 * w.D * flops.n_sel(w.S, w.top_k) * w.Hq * w.B),
    # main-attention backward: S, dP (2d each), dV, dK, dQ (2d each) per selected pair and head
    "attn_bwd": ("tensor", lambda w: 10 * w.D * flops.n_sel(w.S, w.top_k) * w.Hq * w.B),
    # proxy backward: z recompute, dKp, dQp (2d each) per selected pair and proxy head
    "proxy_bwd": ("tensor", lambda w: 6 * w.D * flops.n_sel(w.S, w.top_k) * w.Hp * w.B),
    "proxy_lse": ("tensor", lambda w: 2 * w.D * flops.n_sel(w.S, w.top_k) * w.Hp * w.B),
    # warmup step: the same per-pair work over every causal pair
    "dense_fwd": ("tensor", lambda w: 4 * w.D * flops.n_dense(w.S) * w.Hq * w.B),
    "attn_bwd_dense": ("tensor", lambda w: 10 * w.D * flops.n_dense(w.S) * w.Hq * w.B),
    "proxy_bwd_dense": ("tensor", lambda w: 6 * w.D * flops.n_dense(w.S) * w.Hp * w.B),
    "proxy_lse_dense": ("tensor", lambda w: 2 * w.D * flops.n_dense(w.S) * w.Hp * w.B),
}


def src_hash(*files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_record(kernel, w):
    """DRAM bytes per launch from the committed ncu summary, if it matches this kernel build."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        recs = json.load(f)
    r = recs.get(kernel)
    if not r or r.get("workload") != w.name:
        return None
    if r.get("src_hash") != src_hash(*r.get("src_files", [])):
        return None  # kernel changed since the counters were taken
    return r.get("dram_bytes_per_launch")


def run_ours(args, w, wi):
    from block_sparse_attention_qp_gb300 import binding as msa

    world, rank, local = dist.init("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    msa.load_library()
    x = make_inputs(w, dist.rank_seed(workload_seed(wi), rank))
    names = ("q", "k", "v", "qp", "kp", "dout")
    g = {n: x[n].to(dev) for n in names}
    shape = msa.make_shape(g["q"], g["k"], g["qp"], w.top_k, w.scale)
    dense = w.top_k == 0  # the warmup step: dense causal attention, proxy KL over the prefix
    ws_f = msa.workspace(shape, msa.OP_WARMUP_FORWARD if dense else msa.OP_FORWARD, dev)
    ws_b = msa.workspace(shape, msa.OP_WARMUP_BACKWARD if dense else msa.OP_BACKWARD, dev)

    def full_step(src):
        if dense:
            o, lse = msa.msa_warmup_forward(src["q"], src["k"], src["v"], w.scale, ws=ws_f)
            grads = msa.msa_warmup_backward(src["q"], src["k"], src["v"], src["qp"], src["kp"], o,
                                            lse, src["dout"], w.scale, ws=ws_b)
            return (o,) + tuple(grads)
        o, lse, bi = msa.msa_forward(src["q"], src["k"], src["v"], src["qp"], src["kp"], w.top_k,
                                     w.scale, ws=ws_f)
        grads = msa.msa_backward(src["q"], src["k"], src["v"], src["qp"], src["kp"], o, lse,
                                 src["dout"], bi, w.top_k, w.scale, ws=ws_b)
        return (o, bi) + tuple(grads)

    for _ in range(args.warmup):
        full_step(g)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        msa.profile_begin()
        n0 = msa.launch_count()
        e0.record(stream)
        for _ in range(args.steps):
            full_step(g)
        e1.record(stream)
        torch.cuda.synchronize()
        launches = msa.launch_count() - n0
        prof = msa.profile_end()
    dist.barrier()
    # device status words (bounded waits that gave up, bad indices): must be 0 for a valid run
    dev_status = {"fwd": msa.msa_device_status(ws_f), "bwd": msa.msa_device_status(ws_b)}
    sec = e0.elapsed_time(e1) / 1e3
    sec_max = dist.max_over_ranks(sec, device=dev)
    tok = w.B * w.S
    value = dist.whole_job_rate(tok * args.steps, world, sec_max)
    fl = flops.step_flops(w.B, w.S, w.Hq, w.Hp, w.top_k, w.D)
    tflops = fl["total"] * args.steps * world / sec_max / 1e12
    peaks, peak_src = measured_peaks()

    # dominant kernel and its roofline
    dom = max(prof.items(), key=lambda kv: kv[1][1])
    dname, (dn, dms) = dom
    per_launch_s = dms / dn / 1e3
    lps = dn / args.steps  # launches per step: the kernel may run in passes over sequence chunks
    bound, work = KERNEL_WORK.get(dname, ("tensor", None))
    roof = None
    if work is not None:
        achieved = work(w) / lps / per_launch_s / 1e12  # a step's work spread over its launches
        peak = peaks["bf16_tflops_sustained"]
        roof = {"kernel": dname, "bound": bound, "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic_record(dname, w),
                "ms_per_launch": per_launch_s * 1e3, "launches_per_step": lps,
                "peak_note": f"dense bf16 sustained {peak_src} (kernel timed inside a long step)"}

    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(args, w, g, full_step, dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, wi, args)

    if rank == 0:
        kernels = {k: {"launches_per_step": n / args.steps, "ms_per_step": ms / args.steps}
                   for k, (n, ms) in sorted(prof.items(), key=lambda kv: -kv[1][1])}
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": sec_max / args.steps * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": config_of(w),
                "tflops": tflops,
                "frac_of_dense_bf16_peak": {
                    "burst": tflops / world / peaks["bf16_tflops"],
                    "sustained": tflops / world / peaks["bf16_tflops_sustained"],
                    "note": f"sparse-counted FLOPs, {peak_src}"},
                "flops_per_step": fl,
                "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": launches, "kernels": kernels, "clocks": clk.summary(),
                "device_status": dev_status}
        print(json.dumps(line), flush=True)
    dist.shutdown()


def measure_e2e(args, w, g, full_step, dev):
    """Same step through the public API with host buffers: every step copies its inputs from
    pinned host memory and every result back to pinned host memory inside the timed region.  As
    a training loop would, the copies run on their own streams: the inputs of step s + 1 load
    (into the second of two device buffers) while step s computes, and step s's results are read
    back while step s + 1 computes; events order each copy after what it depends on."""
    names = ("q", "k", "v", "qp", "kp", "dout")
    host = {n: g[n].to("cpu").pin_memory() for n in names}
    dst = [{n: torch.empty_like(g[n]) for n in names} for _ in range(2)]
    outs = full_step(g)
    host_out = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
    h2d = sum(host[n].numel() * host[n].element_size() for n in names)
    d2h = sum(o.numel() * o.element_size() for o in outs)
    steps = max(1, min(args.steps, 10))
    main = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    done = [None, None]  # per input buffer: compute of the last step that read it

    def run(nsteps):
        start = torch.cuda.Event()
        start.record(main)
        s_in.wait_event(start)
        s_out.wait_event(start)
        for step in range(nsteps):
            j = step % 2
            if done[j] is not None:
                s_in.wait_event(done[j])
            with torch.cuda.stream(s_in):
                for n in names:
                    dst[j][n].copy_(host[n], non_blocking=True)
            ready = torch.cuda.Event()
            ready.record(s_in)
            main.wait_event(ready)
            res = full_step(dst[j])
            fin = torch.cuda.Event()
            fin.record(main)
            done[j] = fin
            s_out.wait_event(fin)
            with torch.cuda.stream(s_out):
                for ho, r in zip(host_out, res):
                    ho.copy_(r, non_blocking=True)
                    r.record_stream(s_out)
        end = torch.cuda.Event()
        end.record(s_out)
        main.wait_event(end)

    run(1)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    run(steps)
    e1.record(main)
    torch.cuda.synchronize()
    sec = e0.elapsed_time(e1) / 1e3
    return {"value": w.B * w.S * steps / sec, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps,
            "overlap": "copies on two streams, overlapped with the neighbouring steps' compute"}


def cpu_model():
    """Host CPU model name (lscpu, else /proc/cpuinfo), for the baseline record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() == "Model name":
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def oracle_full_step_single_thread():
    """The oracle on the whole of the smallest workload (msa_s1k: every selection row, every
    forward row, every gradient) on one host thread.  Returns (seconds, tokens)."""
    import oracle

    wi, w1 = workload_by_name("msa_s1k")
    x64 = oracle_inputs(w1, workload_seed(wi))
    saved = oracle.threads()
    oracle.set_threads(1)
    try:
        t0 = time.perf_counter()
        idx, _ = oracle.select(x64["qp"], x64["kp"], w1.top_k, w1.scale)
        oracle.forward(x64["q"], x64["k"], x64["v"], idx, w1.top_k, w1.scale)
        oracle.backward(x64["q"], x64["k"], x64["v"], x64["qp"], x64["kp"], x64["dout"], idx,
                        w1.top_k, w1.scale)
        sec = time.perf_counter() - t0
    finally:
        oracle.set_threads(saved)
    return sec, w1.B * w1.S


def cpu_baseline(w, wi, args):
    import oracle

    oracle.build()
    x64 = oracle_inputs(w, workload_seed(wi))
    rng = np.random.default_rng(1)
    toks = sample_tokens(w, args.ref_tokens, rng)
    sec = oracle_sample(w, x64, idx_builder(w), toks)
    st_sec, st_tok = oracle_full_step_single_thread()
    return {"value": len(toks) / sec, "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"{len(toks)} random tokens of {w.name} (all {w.Hp} groups, {w.Hq} heads): "
                      f"selection rows, forward rows, exact share of every gradient; "
                      f"{sec:.1f} s",
            "single_thread_msa_s1k": {"value": st_tok / st_sec, "unit": UNIT, "sec": st_sec,
                                      "cores": 1, "sample": "the whole msa_s1k step"}}


# ------------------------------------------------------------------------------ decode (inference)
DECODE = dict(name="msa_decode_b128", B=128, ctx=32768, Hq=64, Hkv=8, Hp=8, top_k=16)


def run_decode(args):
    """One decode step per iteration: B sequences, each decoding its next token against caches of
    `ctx` tokens (proxy block scores over the whole proxy-key cache, selection, sparse attention
    over the 16 selected blocks).  Caches are drawn on the device (seeded) -- they are inputs of
    the step, not work inside it.  Memory-bound: reported against the measured copy bandwidth."""
    from block_sparse_attention_qp_gb300 import binding as msa

    c = DECODE
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    msa.load_library()
    gen = torch.Generator(device=dev)
    gen.manual_seed(2001)
    B, S, Hq, Hkv, Hp, D = c["B"], c["ctx"], c["Hq"], c["Hkv"], c["Hp"], 128

    def rnd(*shape):
        return torch.randn(*shape, generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)

    k, v, kp = rnd(B, S, Hkv, D), rnd(B, S, Hkv, D), rnd(B, S, 1, D)
    q, qp = rnd(B, Hq, D), rnd(B, Hp, D)
    seq_len = torch.full((B,), S, dtype=torch.int32, device=dev)
    shape = msa.Shape(B, S, Hq, Hkv, Hp, D, c["top_k"], D ** -0.5)
    ws = msa.workspace(shape, msa.OP_DECODE, dev)

    def step():
        return msa.msa_decode(q, qp, k, v, kp, seq_len, c["top_k"], D ** -0.5, ws=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clk:
        e0.record()
        for _ in range(args.steps):
            step()
        e1.record()
        torch.cuda.synchronize()
    status = msa.msa_device_status(ws)
    sec = e0.elapsed_time(e1) / 1e3 / args.steps
    # per-kernel CUDA-event times, from a separate loop after the timed region
    msa.profile_begin()
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    prof = msa.profile_end()
    kernels = {k: {"launches_per_step": c / args.steps, "ms_per_step": ms / args.steps}
               for k, (c, ms) in sorted(prof.items(), key=lambda kv: -kv[1][1])}
    # bytes one step must read: every proxy-key row before the local block, the selected K and V
    # blocks of every (sequence, KV head), the queries; and write: outputs and selection
    kp_bytes = B * (S - 128) * D * 2
    kv_bytes = B * Hkv * c["top_k"] * 128 * D * 2 * 2
    io_bytes = B * (Hq + Hp) * D * 2 + B * Hq * (D * 2 + 4) + B * Hp * c["top_k"] * 4
    gbs = (kp_bytes + kv_bytes + io_bytes) / sec / 1e9
    peaks, peak_src = measured_peaks()
    line = {"metric": "MSA decode tokens/s (one new token per sequence)", "value": B / sec,
            "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (caches drawn on the device)",
            "config": {"workload": c["name"], "B": B, "context": S, "Hq": Hq, "Hkv": Hkv,
                       "Hp": Hp, "d": D, "top_k": c["top_k"], "block": 128,
                       "l2": f"caches larger than L2 ({(2 * k.numel() + kp.numel()) * 2 / 2**30:.1f} GiB); no flush"},
            "roofline": {"kernel": "decode (scores + selection + attention)", "bound": "hbm",
                         "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "traffic": None,
                         "peak_note": f"copy bandwidth {peak_src}"},
            "gpu_launches": 3 * args.steps, "clocks": clk.summary(), "device_status": status,
            "kernels": kernels}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="msa_s64k_planted")
    ap.add_argument("--ref-tokens", type=int, default=1024)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        print("bench: raising --warmup to the minimum of 3", file=sys.stderr)
        args.warmup = 3
    if args.workload == DECODE["name"]:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the decode mode has no CPU "
                              "reference arm; its parity is tested against the oracle's rows"}))
            return
        run_decode(args)
        return
    wi, w = workload_by_name(args.workload)
    if args.impl == "reference":
        run_reference(args, w, wi)
    else:
        run_ours(args, w, wi)


if __name__ == "__main__":
    main()
