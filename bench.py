"""Throughput of the flow-matching action-expert denoise loop on GB300.

One "step" = one whole pass of the hot path over one batch: ae_bind_prefix of
the batch's prefix KV, then ae_sample with 10 Euler steps.  The headline is
the Pi0.5-shaped batch-1 workload (two 256-token camera slots + 200 text
tokens = 712 valid prefix rows, 18 expert layers, 50 x 32 action chunk); a
batch-16 ragged-prefix line is reported beside it.  All inputs are synthetic
(seeded N(0, sigma), see flow_matching_action_gb300/synth.py).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun each rank runs an independent replica on its own GPU (requests
are independent; there is no collective on the data path); the barrier and the
max over ranks only bracket the timing.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "action chunks/s and µs/flow step (B=1,B=16); % HBM / bf16 tensor roofline"
N_FLOW_STEPS = 10


def algorithmic(dims, n_valid, n_act=None, fp8_weights=False):
    """Algorithmic bytes and flops of ONE flow step (weights read once, prefix
    KV of the valid rows read once per layer; activations neglected).  With
    fp8 weights a block-Linear weight is one byte, plus one fp32 factor per
    weight row."""
    d = dims
    H = d.horizon if n_act is None else n_act
    per_layer_params = (d.q_dim + 2 * d.kv_dim) * d.width + d.width * d.q_dim + 3 * d.mlp * d.width
    weight_bytes = d.layers * per_layer_params * 2
    if fp8_weights:
        rows = (d.q_dim + 2 * d.kv_dim) + d.width + 2 * d.mlp + d.width
        weight_bytes = d.layers * (per_layer_params + 4 * rows)
    kv_bytes = sum(d.layers * 2 * n * d.kv_dim * 2 for n in n_valid)
    B = len(n_valid)
    gemm_flops = 2 * d.layers * per_layer_params * B * H
    attn_flops = sum(4 * d.layers * d.n_q_heads * H * (n + H) * d.head_dim for n in n_valid)
    return weight_bytes + kv_bytes, gemm_flops + attn_flops


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = os.path.join("/tmp", f"ae_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.dev)], stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    mx = float(p[2])
                except ValueError:
                    continue
                for n, v in zip(names, p[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- workloads
def make_workload(name: str, seed: int = 0):
    from flow_matching_action_gb300 import synth
    if name == "pi05_b1":
        return synth.pi05_two_camera(seed, N_FLOW_STEPS)
    if name == "pi05_b16":
        return synth.pi05_batched(seed, N_FLOW_STEPS, 16)
    if name == "pi05_b1_pad2048":
        return synth.pi05_padded(seed, N_FLOW_STEPS, True)
    if name == "tiny":
        return synth.tiny(seed)
    if name == "pi05_shared16":
        return shared_samples(synth.pi05_two_camera(seed, N_FLOW_STEPS), 16, seed)
    if name == "pi05_context":
        return synth.pi05_context(seed, N_FLOW_STEPS)
    raise ValueError(name)


def shared_samples(wl, n_samples, seed):
    """n_samples action samples of the one request of `wl` over its prefix:
    the prefix is laid out once per sample here only so that the oracle and
    the flop count see n_samples requests; the GPU arm binds one copy with
    ae_bind_prefix_shared.  Each sample has its own noise."""
    import dataclasses
    from flow_matching_action_gb300 import synth
    rows = wl.n_rows[0]
    noise = np.stack([synth.request_noise(wl.dims, seed + 100, s) for s in range(n_samples)])
    many = dataclasses.replace(
        wl, name=f"pi05_shared{n_samples}_{rows}", layouts=[list(wl.layouts[0]) for _ in range(n_samples)],
        prefix_k=np.concatenate([wl.prefix_k] * n_samples, axis=1),
        prefix_v=np.concatenate([wl.prefix_v] * n_samples, axis=1),
        mask=np.concatenate([wl.mask] * n_samples), cu_lens=np.arange(n_samples + 1, dtype=np.int32) * rows,
        noise=noise)
    many.shared_rows = rows
    return many


def describe(wl) -> str:
    if wl.context is not None:
        return (f"{wl.name}: Pi0.5-shaped action expert L={wl.dims.layers} D={wl.dims.width} "
                f"F={wl.dims.mlp} Hq={wl.dims.n_q_heads} Hkv={wl.dims.n_kv_heads} dh={wl.dims.head_dim}, "
                f"batch {wl.batch}, prefix as {wl.dims.ctx_dim}-wide per-layer hidden states of "
                f"{min(wl.n_valid)}..{max(wl.n_valid)} valid rows projected into K/V at every bind, "
                f"horizon {wl.dims.horizon} x {wl.dims.action_dim}, {wl.n_steps} Euler steps")
    shared = getattr(wl, "shared_rows", None)
    prefix = (f"{wl.batch} samples over one shared prefix of {shared} rows ({min(wl.n_valid)} valid)"
              if shared is not None else
              f"batch {wl.batch}, valid prefix rows {min(wl.n_valid)}..{max(wl.n_valid)} "
              f"(physical {sum(wl.n_rows)})")
    return (f"{wl.name}: Pi0.5-shaped action expert L={wl.dims.layers} D={wl.dims.width} "
            f"F={wl.dims.mlp} Hq={wl.dims.n_q_heads} Hkv={wl.dims.n_kv_heads} dh={wl.dims.head_dim}, "
            f"{prefix}, horizon {wl.dims.horizon} x {wl.dims.action_dim}, {wl.n_steps} Euler steps")


def _dev(x, dtype):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    return t.to(torch.bfloat16) if dtype == "bf16" else t


# ----------------------------------------------------------------------------- GPU arm
def run_gpu_arm(wl, weights_np, steps, warmup, dist_ctx, measure_e2e=True, stat_reps=50, fp8_weights=False):
    import torch
    from flow_matching_action_gb300 import ae

    dtype = wl.dims.dtype
    dev_w = {k: ([_dev(a, dtype) for a in v] if isinstance(v, list) else _dev(v, dtype))
             for k, v in weights_np.items()}
    stream = torch.cuda.Stream()
    ex = ae.ActionExpert(wl.dims, dev_w, max(wl.batch, 1), max(max(wl.n_rows), 1),
                         stream=stream.cuda_stream, fp8_weights=fp8_weights)
    del dev_w
    shared = getattr(wl, "shared_rows", None)
    rows = shared if shared is not None else None
    context = wl.context is not None
    if context:  # per-layer VLM hidden states, projected into K/V by every bind
        k = _dev(wl.context, dtype)
        v = None
    else:
        k = _dev(wl.prefix_k[:, :rows], dtype)
        v = _dev(wl.prefix_v[:, :rows], dtype)
    mask = torch.from_numpy(wl.mask[:rows]).cuda()
    cu = [int(c) for c in wl.cu_lens]
    rng = np.random.default_rng(123)
    n_noise = 4
    noises = [torch.from_numpy(rng.standard_normal(wl.noise.shape).astype(np.float32)).cuda()
              for _ in range(n_noise)]
    out = torch.empty_like(noises[0])

    def bind():
        if context:
            ex.bind_context(k, cu, mask)
        elif shared is not None:
            ex.bind_prefix_shared(wl.batch, k, v, shared, mask)
        else:
            ex.bind_prefix(k, v, cu, mask)

    def one_step(i):
        bind()
        ex.sample(noises[i % n_noise], wl.n_steps, out)

    with torch.cuda.stream(stream):
        for i in range(warmup):
            one_step(i)
        ex.synchronize()
        info = ex.info()
        launches_per_step = info["launches_last_sample"] + info["launches_last_bind"]

        # -- timed region: device-resident inputs
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        mids = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        clocks = ClockSampler(torch.cuda.current_device())
        dist_ctx.barrier()
        torch.cuda.synchronize()
        clocks.start()
        time.sleep(0.3)  # let the sampler take its first reading
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(steps):
            starts[i].record(stream)
            bind()
            mids[i].record(stream)
            ex.sample(noises[i % n_noise], wl.n_steps, out)
            ends[i].record(stream)
        t1.record(stream)
        torch.cuda.synchronize()
        clk = clocks.stop()
        dist_ctx.barrier()
        total_ms = t0.elapsed_time(t1)
        bind_ms = [starts[i].elapsed_time(mids[i]) for i in range(steps)]
        sample_ms = [mids[i].elapsed_time(ends[i]) for i in range(steps)]
        # per-call statistics (median, p90) over at least stat_reps ae_sample calls
        extra = max(0, stat_reps - steps)
        if extra:
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(extra)]
            bind()
            for i in range(extra):
                ev[i][0].record(stream)
                ex.sample(noises[i % n_noise], wl.n_steps, out)
                ev[i][1].record(stream)
            torch.cuda.synchronize()
            sample_ms = sample_ms + [a.elapsed_time(b) for a, b in ev]

        e2e = None
        if measure_e2e:
            e2e = run_e2e(ex, wl, steps, warmup, stream, dist_ctx)
    ex.close()
    return {"total_ms": total_ms, "bind_ms": bind_ms, "sample_ms": sample_ms, "clocks": clk,
            "launches_per_step": launches_per_step, "e2e": e2e}


def run_e2e(ex, wl, steps, warmup, stream, dist_ctx):
    """The same metric through the public API with HOST buffers: every step copies
    the step's inputs (prefix K/V, mask, noise) from pinned host memory, binds,
    samples, and reads the actions back to pinned host memory."""
    import torch
    dtype = wl.dims.dtype
    hk = torch.from_numpy(np.ascontiguousarray(wl.prefix_k))
    hv = torch.from_numpy(np.ascontiguousarray(wl.prefix_v))
    if dtype == "bf16":
        hk, hv = hk.to(torch.bfloat16), hv.to(torch.bfloat16)
    hk, hv = hk.pin_memory(), hv.pin_memory()
    hmask = torch.from_numpy(wl.mask).pin_memory()
    hnoise = torch.from_numpy(wl.noise).pin_memory()
    hout = torch.empty_like(hnoise).pin_memory()
    dk, dv = torch.empty_like(hk, device="cuda"), torch.empty_like(hv, device="cuda")
    dmask = torch.empty_like(hmask, device="cuda")
    dnoise = torch.empty_like(hnoise, device="cuda")
    dout = torch.empty_like(dnoise)
    cu = [int(c) for c in wl.cu_lens]
    h2d = sum(t.numel() * t.element_size() for t in (hk, hv, hmask, hnoise))
    d2h = hout.numel() * hout.element_size()

    def one():
        dk.copy_(hk, non_blocking=True)
        dv.copy_(hv, non_blocking=True)
        dmask.copy_(hmask, non_blocking=True)
        dnoise.copy_(hnoise, non_blocking=True)
        ex.bind_prefix(dk, dv, cu, dmask)
        ex.sample(dnoise, wl.n_steps, dout)
        hout.copy_(dout, non_blocking=True)

    for _ in range(max(warmup, 1)):
        one()
    torch.cuda.synchronize()
    dist_ctx.barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        one()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = dist_ctx.max(t0.elapsed_time(t1))
    return {"ms": ms, "h2d": h2d, "d2h": d2h}


# ----------------------------------------------------------------------------- CPU oracle
def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def oracle_flow_step_seconds(wl, weights_np, budget_s=12.0, min_runs=1):
    """Time the oracle (as it stands) on single flow steps of the workload until the budget is spent."""
    from oracle import ae_oracle
    times = []
    t_start = time.perf_counter()
    while True:
        t0 = time.perf_counter()
        ae_oracle.sample(wl.dims, weights_np, wl.prefix_k, wl.prefix_v, wl.cu_lens, wl.mask,
                         wl.noise, 1)
        times.append(time.perf_counter() - t0)
        if len(times) >= min_runs and time.perf_counter() - t_start >= budget_s:
            break
    return statistics.median(times), len(times)


def cpu_baseline(wl, weights_np, budget_s=12.0):
    sec, runs = oracle_flow_step_seconds(wl, weights_np, budget_s)
    chunk_s = sec * wl.n_steps
    return {"value": wl.batch / chunk_s, "unit": "chunks/s", "cores": blas_threads(),
            "kind": "oracle",
            "sample": f"{runs} single flow steps of {wl.name} (batch {wl.batch}) through the float64 "
                      f"NumPy oracle, median {sec:.3f} s per flow step, scaled x{wl.n_steps} to a chunk"}


# ----------------------------------------------------------------------------- dist
class DistCtx:
    def __init__(self, n_gpus):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl"
            import torch
            if not torch.cuda.is_available():
                backend = "gloo"
            else:
                torch.cuda.set_device(self.local_rank)
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if self.pg is None:
            return x
        import torch
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], p.get("bf16_tflops_sustained", p["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, 1700.0, "fallback"


# ----------------------------------------------------------------------------- main
def _code_tokens(text: str) -> str:
    """C/C++/CUDA source with its comments removed and whitespace runs collapsed:
    what the compiler sees, so that editing a comment leaves the digest alone."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":  # string or character literal, copied whole
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_digest() -> str:
    """SHA-256 over the code of the CUDA sources and the C header (what the
    kernels are built from), comments and whitespace aside."""
    import glob
    import hashlib
    root = os.path.dirname(os.path.abspath(__file__))
    h = hashlib.sha256()
    files = sorted(glob.glob(os.path.join(root, "flow_matching_action_gb300", "csrc", "*")))
    for p in files + [os.path.join(root, "include", "ae.h")]:
        h.update(os.path.basename(p).encode())
        with open(p, encoding="utf-8", errors="replace") as f:
            h.update(_code_tokens(f.read()).encode())
    return h.hexdigest()


def measured_traffic(workload: str):
    """DRAM bytes per flow step from the committed ncu summary, or None when the
    kernels changed since those counters were taken."""
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_sha256") != source_digest():
        return None
    return rec.get("bytes_per_flow_step", {}).get(workload)


def side_line(name, w, args, dist_ctx, tf_burst, tf_sust, peak_kind, hbm, fp8_weights=False):
    """A workload reported beside the headline one: against the HBM roofline at
    batch 1 (weight streaming), else against the bf16 tensor roofline."""
    wl2 = make_workload(name)
    b2, f2 = algorithmic(wl2.dims, wl2.n_valid, fp8_weights=fp8_weights)
    reps2 = max(args.reps, args.steps)
    if wl2.dims.ctx_dim > 0:
        from flow_matching_action_gb300 import synth
        w = {**w, **synth.make_context_weights(wl2.dims, 0)}
    r2 = run_gpu_arm(wl2, w, reps2, args.warmup, dist_ctx, measure_e2e=False, stat_reps=reps2,
                     fp8_weights=fp8_weights)
    s2 = statistics.median(r2["sample_ms"])
    t2 = dist_ctx.max(r2["total_ms"]) / reps2
    tflops = f2 * wl2.n_steps / (s2 / 1e3) / 1e12
    extra = {}
    if wl2.dims.ctx_dim > 0:
        # the bind projects every valid row of every layer: 2 GEMMs [n, C] x [C, Hkv dh] a layer
        d2 = wl2.dims
        pf = 2.0 * 2 * d2.layers * sum(wl2.n_valid) * d2.ctx_dim * d2.kv_dim
        bm = statistics.median(r2["bind_ms"])
        extra["context_projection"] = {"bind_ms_median": bm, "flops_per_bind": pf,
                                       "achieved_tflops": pf / (bm / 1e3) / 1e12,
                                       "frac_of_burst_bf16": pf / (bm / 1e3) / 1e12 / tf_burst}
    if fp8_weights:
        extra["weights"] = ("block Linears (wq wk wv wo wg wu wd) as per-tensor e4m3 codes, quantized by "
                            "ae_create (AE_WEIGHTS_FP8_E4M3); everything else bf16 / fp32")
    return {**extra, "workload": describe(wl2), "chunks_per_s": wl2.batch / (t2 / 1e3) * dist_ctx.world,
            "ms_per_step": t2, "us_per_flow_step": s2 * 1e3 / wl2.n_steps,
            "sample_ms_median": s2, "sample_ms_p90": float(np.percentile(r2["sample_ms"], 90)),
            "sample_calls_timed": len(r2["sample_ms"]),
            "clocks": r2["clocks"],
            "roofline": ({"bound": "hbm", "achieved": b2 * wl2.n_steps / (s2 / 1e3) / 1e9, "peak": hbm,
                          "unit": "GB/s", "frac": b2 * wl2.n_steps / (s2 / 1e3) / 1e9 / hbm,
                          "algorithmic_bytes_per_flow_step": b2,
                          "traffic": measured_traffic(name + ("_fp8" if fp8_weights else "")),
                          "traffic_unit": "DRAM bytes read + written per flow step (ncu, warm L2)"}
                         if wl2.batch == 1 else
                         {"bound": "tensor", "achieved": tflops, "peak": tf_sust,
                         "unit": "TFLOP/s", "frac": tflops / tf_sust,
                         "peak_burst": tf_burst, "frac_of_burst": tflops / tf_burst,
                         "peak_kind": f"{peak_kind} sustained cuBLAS bf16 (frac); "
                                      f"{peak_kind} burst cuBLAS bf16 (frac_of_burst)",
                         "algorithmic_flops_per_flow_step": f2,
                         "traffic": measured_traffic(name),
                         "traffic_unit": "DRAM bytes read + written per flow step (ncu, warm L2)"})}


def prefill_line(args, dist_ctx, tf_burst, tf_sust, peak_kind):
    """The VLM prefill that produces the prefix KV (ae_prefill): a decoder with
    the widths and depth of Pi0.5's 2B VLM (18 layers, D 2048, MLP 16384, 8 q
    heads, one KV head, head_dim 256) over the 712-token two-camera prefix.
    Its 4 GB of synthetic bf16 weights are drawn on the device (seeded
    torch generator, N(0, 0.02); norm weights N(0, 0.1) in the modulation
    biases, zero modulation weights), not through the host generator."""
    import dataclasses
    import torch
    from flow_matching_action_gb300 import ae, synth
    d = dataclasses.replace(synth.PI05_VLM_2L, layers=18)
    g = torch.Generator(device="cuda").manual_seed(11)
    D, F, L = d.width, d.mlp, d.layers

    def rnd(*shape, std=synth.WEIGHT_STD):
        return (torch.randn(*shape, generator=g, device="cuda") * std).to(torch.bfloat16)
    zero_mod = torch.zeros(3 * D, D, dtype=torch.bfloat16, device="cuda")
    w = {"w_in": rnd(D, d.action_dim), "b_in": rnd(D), "w_t1": rnd(D, D), "b_t1": rnd(D), "w_t2": rnd(D, D),
         "b_t2": rnd(D), "w_mod_f": rnd(2 * D, D), "b_mod_f": rnd(2 * D), "w_out": rnd(d.action_dim, D),
         "b_out": rnd(d.action_dim)}
    shapes = dict(synth.layer_weight_shapes(d))
    for name in synth.LAYER_WEIGHTS:
        w[name] = []
    for _ in range(L):
        for name in synth.LAYER_WEIGHTS:
            if name in ("w_mod1", "w_mod2"):
                w[name].append(zero_mod)
            elif name in ("b_mod1", "b_mod2"):
                w[name].append(torch.cat([rnd(D, std=0.1), torch.zeros(D, dtype=torch.bfloat16, device="cuda"),
                                          torch.ones(D, dtype=torch.bfloat16, device="cuda")]))
            else:
                w[name].append(rnd(*shapes[name]))
    stream = torch.cuda.Stream()
    ex = ae.ActionExpert(d, w, 1, 0, stream=stream.cuda_stream)
    del w
    n = d.horizon
    emb = torch.randn(n, D, generator=g, device="cuda").to(torch.bfloat16)
    k = torch.empty(L, n, d.kv_dim, dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    reps = max(args.reps // 5, 5)
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 1)):
            ae.ae_prefill(ex.ctx, 1, emb, k, v)
        ex.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in ev:
            a.record(stream)
            ae.ae_prefill(ex.ctx, 1, emb, k, v)
            b.record(stream)
        torch.cuda.synchronize()
    launches = ex.info()["launches_last_sample"]
    ex.close()
    ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    per_layer = 2 * n * (d.q_dim + 2 * d.kv_dim) * D
    mlp_o = 2 * n * (D * d.q_dim + 3 * F * D)
    attn = 4 * d.n_q_heads * n * n * d.head_dim
    flops = L * (per_layer + attn) + (L - 1) * mlp_o  # the last layer stops after its K/V
    tflops = flops / (ms / 1e3) / 1e12
    return {"workload": f"VLM prefill: L={L} D={D} F={F} Hq={d.n_q_heads} Hkv={d.n_kv_heads} dh={d.head_dim}, "
                        f"one request of {n} prefix tokens -> per-layer K/V",
            "ms_per_prefill": ms, "prefills_timed": reps, "gpu_launches": launches,
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": tf_burst, "unit": "TFLOP/s",
                         "frac": tflops / tf_burst, "peak_kind": f"{peak_kind} burst cuBLAS bf16",
                         "algorithmic_flops": flops}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="pi05_b1")
    ap.add_argument("--batched", default="pi05_b16", help="second workload reported beside ('' = none)")
    ap.add_argument("--shared", default="pi05_shared16",
                    help="many samples over one shared prefix, reported beside ('' = none)")
    ap.add_argument("--no-prefill", action="store_true", help="skip the VLM prefill line")
    ap.add_argument("--context", default="pi05_context",
                    help="prefix as per-layer VLM hidden states projected at bind, reported beside ('' = none)")
    ap.add_argument("--weights", default="bf16", choices=["bf16", "fp8"],
                    help="block-Linear weights of the headline workload (fp8: AE_WEIGHTS_FP8_E4M3)")
    ap.add_argument("--fp8", default="pi05_b1",
                    help="workload also run with e4m3 block-Linear weights ('' = none)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--reps", type=int, default=50, help="minimum ae_sample calls in the per-call statistics")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("note: fewer than 3 warm-up steps", file=sys.stderr)

    dist_ctx = DistCtx(args.gpus)
    from flow_matching_action_gb300 import synth
    wl = make_workload(args.workload)
    w = synth.make_weights(wl.dims, 0)
    fp8_main = args.weights == "fp8"
    bytes_fs, flops_fs = algorithmic(wl.dims, wl.n_valid, fp8_weights=fp8_main)

    if args.impl == "reference":
        if dist_ctx.rank != 0:
            dist_ctx.close()
            return
        for _ in range(args.warmup):
            pass  # the oracle has no warm-up state; its first run is timed like the rest
        # one step = one flow step of the workload through the oracle (measured);
        # a chunk is n_steps of them, so the chunks/s value divides by n_steps
        per = []
        for _ in range(args.steps):
            sec, _ = oracle_flow_step_seconds(wl, w, budget_s=0.0)
            per.append(sec)
        ms = statistics.median(per) * 1e3
        value = wl.batch / (ms * wl.n_steps / 1e3)
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "chunks/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                "step": f"one flow step of {wl.name} through the oracle (a chunk = {wl.n_steps} flow steps)",
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": {"workload": describe(wl)},
                "cpu_baseline": {"value": value, "unit": "chunks/s", "cores": blas_threads(),
                                 "kind": "oracle",
                                 "sample": f"each step: one flow step of {wl.name} through the float64 "
                                           f"NumPy oracle, scaled x{wl.n_steps} to a chunk"},
                "e2e": {"value": value, "unit": "chunks/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        dist_ctx.close()
        return

    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (sm_103a); the product has no CPU path")
    torch.cuda.set_device(dist_ctx.local_rank)
    from flow_matching_action_gb300 import build as ae_build
    if dist_ctx.rank == 0:
        ae_build.build()
    dist_ctx.barrier()
    ae_build.build()

    res = run_gpu_arm(wl, w, args.steps, args.warmup, dist_ctx, measure_e2e=not args.no_e2e,
                      stat_reps=args.reps, fp8_weights=fp8_main)
    total_ms = dist_ctx.max(res["total_ms"])
    ms_per_step = total_ms / args.steps
    chunks = wl.batch * args.steps * dist_ctx.world
    value = chunks / (total_ms / 1e3)
    sample_ms = statistics.median(res["sample_ms"])
    bind_ms = statistics.median(res["bind_ms"])
    hbm, tf_burst, tf_sust, peak_kind = peaks()
    # roofline of the dominant launch: the whole ae_sample call (10 flow steps)
    achieved_gbs = bytes_fs * wl.n_steps / (sample_ms / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "chunks/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,0.02) weights, N(0,1) prefix KV and noise)",
        "config": {"workload": describe(wl), "batch": wl.batch, "valid_prefix_rows": wl.n_valid,
                   "n_flow_steps": wl.n_steps, "step": "ae_bind_prefix + ae_sample(10 Euler steps)",
                   "l2": ("inputs larger than L2: 311 MB of e4m3 block-Linear weights streamed per flow step"
                          if fp8_main else "inputs larger than L2: 623 MB of bf16 weights streamed per flow step"),
                   "weights": "e4m3 block Linears (AE_WEIGHTS_FP8_E4M3)" if fp8_main else "bf16",
                   "parallelism": f"replicas x{dist_ctx.world}"},
        "us_per_flow_step": sample_ms * 1e3 / wl.n_steps,
        "sample_ms_median": sample_ms, "sample_ms_p90": float(np.percentile(res["sample_ms"], 90)),
        "sample_calls_timed": len(res["sample_ms"]),
        "bind_ms_median": bind_ms,
        "roofline": {"kernel": "ae_sample (all its launches, one flow step = 1 unit)",
                     "bound": "hbm", "achieved": achieved_gbs, "peak": hbm, "unit": "GB/s",
                     "frac": achieved_gbs / hbm,
                     "traffic": measured_traffic(args.workload + ("_fp8" if fp8_main else "")),
                     "traffic_unit": "DRAM bytes read + written per flow step (ncu, warm L2)",
                     "peak_kind": f"{peak_kind} HBM copy bandwidth",
                     "algorithmic_bytes_per_flow_step": bytes_fs},
        "clocks": res["clocks"],
        "gpu_launches": int(res["launches_per_step"] * args.steps),
    }
    if res["e2e"] is not None:
        e = res["e2e"]
        line["e2e"] = {"value": chunks / (e["ms"] / 1e3), "unit": "chunks/s",
                       "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"]}
    for key, name in (("batched", args.batched), ("shared_prefix", args.shared), ("context", args.context)):
        if name:
            line[key] = side_line(name, w, args, dist_ctx, tf_burst, tf_sust, peak_kind, hbm)
    if args.fp8:
        line["fp8_weights"] = side_line(args.fp8, w, args, dist_ctx, tf_burst, tf_sust, peak_kind, hbm,
                                        fp8_weights=True)
    if not args.no_prefill:
        line["prefill"] = prefill_line(args, dist_ctx, tf_burst, tf_sust, peak_kind)
    if dist_ctx.rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, w)
    if dist_ctx.rank == 0:
        print(json.dumps(line))
    dist_ctx.close()


if __name__ == "__main__":
    main()
