"""Benchmark of the GB300 MoE FFN block: canvas-tokens/s per layer forward.

Workload: one DiffusionGemma MoE feed-forward layer over a 256-token canvas
(hidden 2816, 128 experts top-8, expert FFN 704, dense FFN 2112, bf16
weights N(0, 0.02), activations N(0, 1), seed 1; synthetic).  A step is one
whole forward of the block (router, grouping, gate_up, down, combine) on
that canvas with inputs resident in HBM.  The 1.56 GB of weights read per
step are 12x the L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload canvas256|canvas256_q4|canvas256_q4d8|batch2048_zipf|stack30_q4|
                              sc_canvas256|sc_canvas256_q4|sc_canvas256_q8]

Prints one JSON line.  ``--impl reference`` times the CPU oracle (the only
reference there is: the pages hold no runnable implementation) on the host
cores, on a bounded token sample per step.
"""

from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "canvas-tokens/s per MoE layer (µs/layer) and % of HBM/tensor roofline, 1 GB300"
UNIT = "canvas-tokens/s"
WORKLOAD = "canvas256"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def workload_desc(wl):
    if wl.quant:
        fm = lambda b: "NVFP4 (e2m1, e4m3 per 16, fp32 per matrix)" if b == 16 else f"group-64 affine {b}-bit"
        wdesc = (f"N(0,{wl.weight_std}) draws in {fm(wl.quant[0])} (experts), "
                 f"{fm(wl.quant[1])} (dense), {fm(wl.quant[2])} (router)")
    else:
        wdesc = f"bf16 weights N(0,{wl.weight_std})"
    extra = f", Zipf router bias beta {wl.zipf_beta}" if wl.zipf_beta else ""
    return (f"{wl.name}: one DiffusionGemma MoE FFN layer, T={wl.tokens} tokens "
            f"({wl.tokens // 256} canvas{'es' if wl.tokens > 256 else ''}), "
            f"H={wl.hidden}, E={wl.n_experts} top-{wl.top_k}, expert FFN {wl.expert_inter}, "
            f"dense FFN {wl.dense_inter}, {wdesc}{extra}, seed {wl.seed}")


def weight_bytes(n, bits):
    """Bytes of n weights: bf16, group-64 affine codes plus a bf16 scale and
    bias per 64 weights, or NVFP4 (bits code 16) codes plus an e4m3 scale per
    16 weights."""
    if bits == 16:
        return n // 2 + n // 16
    return 2 * n if bits is None else n * bits // 8 + n // 64 * 4


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def code_digest(paths):
    """sha256 (16 hex digits) of the sources with comments and whitespace
    removed: it changes when the compiled code can, not when a comment does."""
    import hashlib
    import re
    h = hashlib.sha256()
    for path in paths:
        src = open(path).read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(re.sub(r"\s+", "", src).encode())
    return h.hexdigest()[:16]


def gate_up_traffic():
    """DRAM bytes per gate_up launch from the committed ncu capture, while the
    GEMM sources are the ones it was taken on (None otherwise)."""
    path = os.path.join(ROOT, "profiles", "gemm_gate_up_canvas256.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path))
    csrc = os.path.join(ROOT, "moe_expert_ffn_dg_gb300", "csrc")
    digest = code_digest([os.path.join(csrc, f) for f in rec["hashed_sources"]])
    return rec["dram_bytes_per_launch"] if digest == rec["gemm_code_digest"] else None


def traffic_for(wl):
    return gate_up_traffic() if wl.name == WORKLOAD else None


def algorithmic(wl, counts):
    """Algorithmic bytes and FLOPs of one layer forward and of its gate_up
    GEMM: weights of the experts that received tokens, dense and router
    weights, the activation read and the output write; intermediates that
    an ideal kernel keeps on chip are not counted.  FLOPs exclude padding."""
    T, H, E, K, I, D = wl.tokens, wl.hidden, wl.n_experts, wl.top_k, wl.expert_inter, wl.dense_inter
    eb, db, rb = wl.quant if wl.quant else (None, None, None)
    touched = int((np.asarray(counts) > 0).sum())
    gu_w = touched * weight_bytes(2 * I * H, eb) + weight_bytes(2 * D * H, db)
    dn_w = touched * weight_bytes(H * I, eb) + weight_bytes(H * D, db)
    router_w = weight_bytes(E * H, rb)
    layer_bytes = gu_w + dn_w + router_w + 2 * T * H * 2 + 4 * H * 2 + E * 2
    layer_flops = 2 * T * H * E + 2 * T * K * 3 * H * I + 2 * T * 3 * H * D
    gu_bytes = gu_w + T * K * H * 2 + T * H * 2 + T * K * I * 2 + T * D * 2
    return {"touched_experts": touched, "layer_bytes": layer_bytes, "layer_flops": layer_flops,
            "gate_up_bytes": gu_bytes}


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.flush()
        rows = [r.split(",") for r in open(self.f.name).read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            try:
                sm.append(float(r[1]))
                smax = float(r[2])
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_baseline(wl, p, h, max_seconds=30.0):
    """The fp64 oracle, as it stands, on a bounded token sample of the same
    workload (tokens are independent, so a sample times the per-token cost)."""
    import oracle
    t0 = time.time()
    n = 16
    oracle.moe_block_forward(h[:n], p, wl.top_k, wl.expert_inter, with_perm=False)
    dt = time.time() - t0
    # grow the sample while it stays inside the time budget
    while n < wl.tokens and dt * 2 * 1.2 < max_seconds:
        n = min(wl.tokens, n * 2)
        t0 = time.time()
        oracle.moe_block_forward(h[:n], p, wl.top_k, wl.expert_inter, with_perm=False)
        dt = time.time() - t0
    return {"value": n / dt, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{n} of the {wl.tokens} canvas tokens, one layer, fp64 numpy oracle "
                      f"(OpenBLAS threads = host cores), {dt:.2f} s"}


def run_reference(args):
    """The reference arm: the CPU oracle timed on the host cores."""
    import moe_inputs as mi
    import oracle
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    wl = mi.get_workload(args.workload)
    if wl.name.startswith("sc_"):
        p = mi.make_sc_inputs(wl, randvec=True)
        n, dt = sc_cpu_sample(wl, p, 120.0)
        line = {"impl": "reference", "metric": SC_METRIC, "value": n / dt, "unit": UNIT,
                "n_gpus": args.gpus, "steps": 1, "warmup": 0, "ms_per_step": 1000.0 * dt,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": {"workload": sc_desc(wl), "tokens_per_step": n},
                "cpu_baseline": {"value": n / dt, "unit": UNIT, "cores": os.cpu_count(),
                                 "kind": "oracle", "sample": f"{n} canvas tokens, fp64 oracle"},
                "e2e": {"value": n / dt, "unit": UNIT, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return
    p = mi.make_layer_inputs(wl)
    h = mi.make_tokens(wl)
    # decode the weights to float64 once, outside the timed steps; the
    # oracle accepts float64 weights as they are
    pf = dict(p)
    for k in ("router", "gate_up", "down", "dense_gate", "dense_up", "dense_down"):
        pf[k] = oracle.to_f64(p[k])
    # one token per step, bounded to about two minutes in total
    t0 = time.time()
    oracle.moe_block_forward(h[:1], pf, wl.top_k, wl.expert_inter, with_perm=False)
    one = max(time.time() - t0, 1e-4)
    steps = max(1, min(args.steps, int(120.0 / one)))
    for i in range(min(args.warmup, 3)):
        oracle.moe_block_forward(h[i:i + 1], pf, wl.top_k, wl.expert_inter, with_perm=False)
    t0 = time.time()
    for i in range(steps):
        j = i % wl.tokens
        oracle.moe_block_forward(h[j:j + 1], pf, wl.top_k, wl.expert_inter, with_perm=False)
    dt = time.time() - t0
    value = steps / dt
    sample = (f"{steps} steps of 1 canvas token each (of {args.steps} requested; bounded to "
              f"~2 min), fp64 numpy oracle, weights decoded to float64 before timing")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": steps, "warmup": args.warmup, "ms_per_step": 1000.0 * dt / steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": workload_desc(wl), "tokens_per_step": 1},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def _gen_layer(job):
    """Worker of the weight-generation pool: one layer's seeded draws."""
    import moe_inputs as mi
    name, layer = job
    return layer, mi.make_layer_inputs(mi.get_workload(name), layer=layer)


def run_stack(args):
    """The 30-layer 4-bit stack over 64 canvases (16384 tokens): a step is one
    forward through all layers (each with its own seeded weights), timed as a
    whole and reported per layer."""
    import multiprocessing as mp

    import moe_inputs as mi
    wl = mi.get_workload(args.workload)
    L = wl.n_layers
    # generate the layers' weights on the host cores before any CUDA call
    t_gen = time.time()
    ctx = mp.get_context("spawn")
    pool = ctx.Pool(processes=max(1, min(16, (os.cpu_count() or 2) - 1)))
    gen = pool.imap(_gen_layer, [(wl.name, l) for l in range(L)])

    import torch

    import moe_expert_ffn_dg_gb300 as pkg
    from moe_expert_ffn_dg_gb300 import binding as B
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    pkg.build()
    pkg.load_library()
    eb, db, rb = wl.quant
    fmt = {4: B.DG_FMT_AFFINE_U4_G64, 8: B.DG_FMT_AFFINE_U8_G64}
    shape = dict(hidden=wl.hidden, n_experts=wl.n_experts, top_k=wl.top_k,
                 expert_inter=wl.expert_inter, dense_inter=wl.dense_inter, max_tokens=wl.tokens)
    ws = torch.empty(pkg.MoEBlock.workspace_bytes(**shape, expert_fmt=fmt[eb], dense_fmt=fmt[db],
                                                  router_fmt=fmt[rb]), dtype=torch.uint8, device=dev)
    blocks, scalars, p0 = [None] * L, [None] * L, None
    for layer, p in gen:
        blocks[layer] = pkg.MoEBlock.from_params(p, **shape, device=dev, workspace=ws)
        scalars[layer] = p["layer_scalar"]
        if layer == 0:
            p0 = p
    pool.close()
    pool.join()
    t_gen = time.time() - t_gen
    h_np = mi.make_tokens(wl)
    h = torch.from_numpy(h_np.view(np.int16)).to(dev).view(torch.bfloat16)
    bufs = [torch.empty_like(h), torch.empty_like(h)]
    stream = torch.cuda.current_stream(dev)

    def step(x):
        for l in range(L):
            out = bufs[l % 2]
            blocks[l].forward(x, scalars[l], out=out)
            x = out
        return x

    for _ in range(max(args.warmup, 3)):
        step(h)
    torch.cuda.synchronize(dev)
    st = blocks[0].device_status()
    if st[0] != 0:
        raise RuntimeError(f"device status after warm-up: {st}")
    names = B.dg_moe_kernel_names(blocks[0].handle)
    nk = len(names)
    prof_layer = L // 2
    elapsed_ms, clk = time_steps(lambda: step(h), stream, dev, args.steps)
    st = blocks[0].device_status()
    if st[0] != 0:
        raise RuntimeError(f"device status after timing: {st}")
    ms_step = elapsed_ms / args.steps
    per_kernel_us = kernel_split(blocks[prof_layer], lambda: step(h), stream, dev,
                                 max(3, min(args.steps, 20)), B.dg_moe_set_profile_events, names)

    # end to end: pinned host input -> device, all layers, output -> host
    h_host = torch.from_numpy(h_np.view(np.int16)).view(torch.bfloat16).pin_memory()
    o_host = torch.empty_like(h_host).pin_memory()
    e2e_steps = max(3, min(args.steps, 10))
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        x = h_host.to(dev, non_blocking=True)
        o_host.copy_(step(x), non_blocking=True)
        torch.cuda.synchronize(dev)
    e2e_s = (time.perf_counter() - t0) / e2e_steps

    _, dbg = blocks[0].forward(h, scalars[0], debug=True)
    counts = np.diff(dbg["offsets"].cpu().numpy())
    alg = algorithmic(wl, counts)
    hbm, bf16_burst, bf16_sus, src = peaks()
    T, H, K, I, D = wl.tokens, wl.hidden, wl.top_k, wl.expert_inter, wl.dense_inter
    gu_flops = 2 * T * K * H * 2 * I + 2 * T * H * 2 * D
    gu = names.index("gemm_gate_up")
    gu_tf = gu_flops / (per_kernel_us[gu] * 1e-6) / 1e12
    t_layer = ms_step / L / 1000.0
    line = {
        "metric": METRIC, "value": T / t_layer, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_desc(wl) + f", {L} layers each with its own weights",
                   "tokens_per_step": T, "layers_per_step": L, "us_per_layer": t_layer * 1e6,
                   "weights": f"u{eb} g64 affine experts and dense, u{rb} router, dequantised "
                              f"to bf16 on chip", "weight_generation_s": round(t_gen, 1),
                   "l2": f"no flush: {alg['layer_bytes'] / 1e9:.3f} GB of weights per layer, "
                         f"{alg['layer_bytes'] / 129e6:.1f}x the 129 MB L2"},
        "roofline": {"bound": "tensor", "kernel": "gemm_gate_up", "achieved": gu_tf,
                     "peak": bf16_sus, "unit": "TFLOP/s", "frac": gu_tf / bf16_sus, "traffic": None,
                     "peak_source": f"{src} (MEASURED_PEAKS.json bf16_tflops_sustained)",
                     "algorithmic_flops_per_launch": gu_flops, "us_per_launch": per_kernel_us[gu],
                     "kernel_of_layer": prof_layer},
        "layer_roofline": {"bytes": alg["layer_bytes"], "flops": alg["layer_flops"],
                           "achieved_tflops": alg["layer_flops"] / t_layer / 1e12,
                           "frac_of_bf16_peak": alg["layer_flops"] / t_layer / 1e12 / bf16_sus,
                           "basis": f"flops / {bf16_sus} TF/s ({src}, sustained)"},
        "kernels_us": {n: round(float(v), 3) for n, v in zip(names, per_kernel_us)},
        "e2e": {"value": T * L / e2e_s, "unit": UNIT, "h2d_bytes_per_step": int(h_host.numel() * 2),
                "d2h_bytes_per_step": int(o_host.numel() * 2), "steps": e2e_steps,
                "note": "per layer: tokens / (end-to-end step time / layers)"},
        "clocks": clk,
        "gpu_launches": launches_per_forward(wl, nk) * L * args.steps,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, p0, h_np, max_seconds=20.0)
    for b in blocks:
        b.close()
    print(json.dumps(line))


SC_METRIC = "canvas-tokens/s of the self-conditioning MLP (µs/call) and % of HBM roofline, 1 GB300"


def sc_desc(wl):
    w = (f"gate/up/down N(0,{wl.weight_std}) draws in group-64 affine {wl.quant[1]}-bit"
         if wl.quant else f"bf16 gate/up/down N(0,{wl.weight_std})")
    return (f"{wl.name}: the self-conditioning MLP of DiffusionGemma (pre-normed GEGLU of the "
            f"dense FFN's shape on the soft signal, added to the embeddings, weightless "
            f"RMSNorm), T={wl.tokens} tokens, H={wl.hidden}, FFN {wl.dense_inter}, {w}, "
            f"embeddings and signal N(0,1), pre_norm U(0.5,1.5), seed {wl.seed}")


def sc_algorithmic(wl):
    """Bytes and FLOPs of one self-conditioning forward and of its gate_up
    GEMM: the three weight matrices, the embeddings and signal read, the
    output write; x, act and the f32 MLP output stay on chip in an ideal
    kernel."""
    T, H, D = wl.tokens, wl.hidden, wl.dense_inter
    db = wl.quant[1] if wl.quant else None
    w = weight_bytes(3 * D * H, db)
    return {"bytes": w + 3 * T * H * 2 + H * 2, "flops": 2 * T * 3 * H * D,
            "gate_up_bytes": weight_bytes(2 * D * H, db) + T * H * 2 + T * D * 2,
            "gate_up_flops": 2 * T * 2 * H * D}


def sc_cpu_sample(wl, p, max_seconds):
    import oracle
    n, dt = 1, 0.0
    while True:
        t0 = time.time()
        oracle.sc_mlp_forward(p["embeds"][:n], p["signal"][:n], p)
        dt = time.time() - t0
        if n >= wl.tokens or dt * 2 * 1.2 > max_seconds:
            return n, dt
        n = min(wl.tokens, n * 2)


def run_sc(args):
    """The self-conditioning MLP over one canvas: a step is one forward
    (pre-norm, gate_up + GEGLU, down, residual + RMSNorm) with the inputs
    resident in HBM."""
    import torch

    import moe_expert_ffn_dg_gb300 as pkg
    import moe_inputs as mi
    from moe_expert_ffn_dg_gb300 import binding as B
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    pkg.build()
    pkg.load_library()
    wl = mi.get_workload(args.workload, **({"tokens": args.tokens} if args.tokens else {}))
    p = mi.make_sc_inputs(wl, randvec=True)
    sc = pkg.ScMlp.from_params(p, hidden=wl.hidden, inter=wl.dense_inter, max_tokens=wl.tokens,
                               device=dev)

    def dev16(a):
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)

    e, sig = dev16(p["embeds"]), dev16(p["signal"])
    out = torch.empty_like(e)
    stream = torch.cuda.current_stream(dev)
    names = B.dg_sc_mlp_kernel_names(sc.handle)
    nk = len(names)
    for _ in range(max(args.warmup, 3)):
        sc.forward(e, sig, out=out)
    torch.cuda.synchronize(dev)
    if sc.device_status() != 0:
        raise RuntimeError("device status after warm-up")
    elapsed_ms, clk = time_steps(lambda: sc.forward(e, sig, out=out), stream, dev, args.steps)
    if sc.device_status() != 0:
        raise RuntimeError("device status after timing")
    ms = elapsed_ms / args.steps
    per_kernel_us = kernel_split(sc, lambda: sc.forward(e, sig, out=out), stream, dev,
                                 max(3, min(args.steps, 200)), B.dg_sc_mlp_set_profile_events,
                                 names)

    # end to end: pinned host embeddings and signal in, output back, synchronised
    e_host = torch.from_numpy(p["embeds"].view(np.int16)).view(torch.bfloat16).pin_memory()
    s_host = torch.from_numpy(p["signal"].view(np.int16)).view(torch.bfloat16).pin_memory()
    o_host = torch.empty_like(e_host).pin_memory()
    e_dev, s_dev = torch.empty_like(e), torch.empty_like(sig)
    e2e_steps = max(10, min(args.steps, 2000))
    for i in range(3 + e2e_steps):
        if i == 3:
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
        e_dev.copy_(e_host, non_blocking=True)
        s_dev.copy_(s_host, non_blocking=True)
        sc.forward(e_dev, s_dev, out=e_dev)
        o_host.copy_(e_dev, non_blocking=True)
        torch.cuda.synchronize(dev)
    e2e_s = time.perf_counter() - t0

    alg = sc_algorithmic(wl)
    hbm, bf16_burst, bf16_sus, src = peaks()
    gu = names.index("gemm_gate_up")
    achieved = alg["gate_up_bytes"] / (per_kernel_us[gu] * 1e-6) / 1e9
    t_roof = max(alg["bytes"] / (hbm * 1e9), alg["flops"] / (bf16_burst * 1e12))
    line = {
        "metric": SC_METRIC, "value": wl.tokens / (ms / 1000.0), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": sc_desc(wl), "tokens_per_step": wl.tokens, "us_per_call": ms * 1e3,
                   "l2": f"no flush: inputs and weights resident; {alg['bytes'] / 1e6:.1f} MB per "
                         f"step fit the 129 MB L2, so the HBM fraction is an upper bound"},
        "roofline": {"bound": "hbm", "kernel": "gemm_gate_up", "achieved": achieved, "peak": hbm,
                     "unit": "GB/s", "frac": achieved / hbm, "traffic": None,
                     "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)",
                     "algorithmic_bytes_per_launch": alg["gate_up_bytes"],
                     "us_per_launch": per_kernel_us[gu]},
        "step_roofline": {"bytes": alg["bytes"], "flops": alg["flops"], "t_roof_us": t_roof * 1e6,
                          "frac": t_roof / (ms / 1000.0),
                          "basis": f"max(bytes / {hbm} GB/s, flops / {bf16_burst} TF/s) ({src})"},
        "kernels_us": {n: round(float(v), 3) for n, v in zip(names, per_kernel_us)},
        "e2e": {"value": wl.tokens * e2e_steps / e2e_s, "unit": UNIT,
                "h2d_bytes_per_step": int(e_host.numel() * 2 + s_host.numel() * 2),
                "d2h_bytes_per_step": int(o_host.numel() * 2), "steps": e2e_steps},
        "clocks": clk,
        "gpu_launches": nk * args.steps,
    }
    if not args.no_cpu_baseline:
        n, dt = sc_cpu_sample(wl, p, 20.0)
        line["cpu_baseline"] = {"value": n / dt, "unit": UNIT, "cores": os.cpu_count(),
                                "kind": "oracle",
                                "sample": f"{n} of the {wl.tokens} canvas tokens, fp64 numpy "
                                          f"oracle, {dt:.2f} s"}
    sc.close()
    print(json.dumps(line))


def time_steps(fwd, stream, dev, steps, local=0, dist=None):
    """Wall time of `steps` back-to-back forwards on the device (CUDA events
    on the launching stream, nothing recorded between the kernels), with
    nvidia-smi clocks sampled meanwhile.  Returns (elapsed ms, clocks)."""
    import torch
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    start.record(stream)
    for _ in range(steps):
        fwd()
    stop.record(stream)
    torch.cuda.synchronize(dev)
    return start.elapsed_time(stop), clocks.stop()


def kernel_split(blk, fwd, stream, dev, steps, set_events, names):
    """Average device time of each kernel of a forward, from a separate pass
    with an event recorded between consecutive kernels (the events stop the
    kernels' programmatic overlap, so these times are a little longer than
    the kernels take inside an event-free step)."""
    import torch
    nk = len(names)
    ev_sets = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)] for _ in range(steps)]
    # torch creates the CUDA event at its first record(): record every event
    # once so the handles given to the library are real
    for evs in ev_sets:
        for e in evs:
            e.record(stream)
    torch.cuda.synchronize(dev)
    for evs in ev_sets:
        set_events(blk.handle, [e.cuda_event for e in evs])
        fwd()
    torch.cuda.synchronize(dev)
    set_events(blk.handle, None)
    per_kernel = np.zeros(nk)
    for evs in ev_sets:
        per_kernel += [evs[j].elapsed_time(evs[j + 1]) for j in range(nk)]
    return per_kernel / len(ev_sets) * 1000.0


ROUTER_TC_MIN_TOKENS = 1024  # the library's tensor-core router threshold


def launches_per_forward(wl, nk):
    # an 8-bit dense branch beside 4-bit experts adds a dense-only launch to
    # each of the two GEMM slots; from 1024 tokens the router slot holds two
    # launches (prep and the router GEMM) and so does the selection slot (fast
    # pass and re-check pass)
    return (nk + (2 if wl.quant and wl.quant[1] != wl.quant[0] else 0)
            + (2 if wl.tokens >= ROUTER_TC_MIN_TOKENS else 0))


def measure_layer(wl, p, h_np, dev, steps, warmup, local=0, neighbours=False, dist=None,
                  budget_s=None):
    """Time one MoE layer on its workload: an event-free pass for the step
    time, a separate pass for the per-kernel split, the routing of the timed
    tokens for the touched-expert count, and the roofline fractions.
    Returns (result dict, block, forward closure)."""
    import torch

    import moe_expert_ffn_dg_gb300 as pkg
    import moe_inputs as mi
    from moe_expert_ffn_dg_gb300 import binding as B
    from moe_expert_ffn_dg_gb300 import replicas

    blk = pkg.MoEBlock.from_params(p, hidden=wl.hidden, n_experts=wl.n_experts, top_k=wl.top_k,
                                   expert_inter=wl.expert_inter, dense_inter=wl.dense_inter,
                                   max_tokens=wl.tokens, device=dev)
    h = torch.from_numpy(h_np.view(np.int16)).to(dev).view(torch.bfloat16)
    out = torch.empty_like(h)
    stream = torch.cuda.current_stream(dev)
    names = B.dg_moe_kernel_names(blk.handle)
    ls = float(p.get("layer_scalar", 1.0))
    if neighbours:
        # the decoder layer's neighbours fused in: h is the layer input, attn
        # the attention output (N(0, 4)), norm weights U(0.5, 1.5)
        g = np.random.default_rng(wl.seed + 200)
        dbf = lambda a: torch.from_numpy(mi.f32_to_bf16_bits(a.astype(np.float32)).view(np.int16)).to(dev).view(torch.bfloat16)
        attn = dbf(g.standard_normal((wl.tokens, wl.hidden)) * 4.0)
        w_pa, w_next = dbf(g.uniform(0.5, 1.5, wl.hidden)), dbf(g.uniform(0.5, 1.5, wl.hidden))
        nxt = torch.empty_like(h)

    def fwd():
        if neighbours:
            blk.forward_neighbours(h, attn, w_pa, w_next, ls, out=out, next_in=nxt)
        else:
            blk.forward(h, ls, out=out)

    t0 = time.perf_counter()
    for _ in range(max(warmup, 3)):
        fwd()
    torch.cuda.synchronize(dev)
    t_warm = (time.perf_counter() - t0) / max(warmup, 3)
    st = blk.device_status()
    if st[0] != 0:
        raise RuntimeError(f"{wl.name}: device status after warm-up: {st}")
    if budget_s:
        steps = max(10, min(steps, int(budget_s / max(t_warm, 1e-6))))
    elapsed_ms, clk = time_steps(fwd, stream, dev, steps, local, dist)
    elapsed_ms = replicas.max_over_ranks(elapsed_ms, dist, dev)
    st = blk.device_status()
    if st[0] != 0:
        raise RuntimeError(f"{wl.name}: device status after timing: {st}")
    ms = elapsed_ms / steps
    per_kernel_us = kernel_split(blk, fwd, stream, dev, max(3, min(steps, 200)),
                                 B.dg_moe_set_profile_events, names)
    # routing of the timed tokens (for the touched-expert count)
    _, dbg = blk.forward(h, ls, debug=True)
    counts = np.diff(dbg["offsets"].cpu().numpy())
    alg = algorithmic(wl, counts)
    if neighbours:
        alg["layer_bytes"] += 2 * wl.tokens * wl.hidden * 2 + 2 * wl.hidden * 2  # attn in, next_in out
    hbm, bf16_burst, bf16_sus, src = peaks()
    T, H, K, I, D = wl.tokens, wl.hidden, wl.top_k, wl.expert_inter, wl.dense_inter
    gu = names.index("gemm_gate_up")
    gu_s = per_kernel_us[gu] * 1e-6
    t_roof = max(alg["layer_bytes"] / (hbm * 1e9), alg["layer_flops"] / (bf16_sus * 1e12))
    gu_flops = 2 * T * K * H * 2 * I + 2 * T * H * 2 * D
    tensor_bound = alg["layer_flops"] / (bf16_sus * 1e12) > alg["layer_bytes"] / (hbm * 1e9)
    if tensor_bound:
        achieved = gu_flops / gu_s / 1e12
        roof = {"bound": "tensor", "kernel": "gemm_gate_up", "achieved": achieved,
                "peak": bf16_sus, "unit": "TFLOP/s", "frac": achieved / bf16_sus, "traffic": None,
                "peak_source": f"{src} (MEASURED_PEAKS.json bf16_tflops_sustained)",
                "algorithmic_flops_per_launch": gu_flops, "us_per_launch": per_kernel_us[gu]}
    else:
        achieved = alg["gate_up_bytes"] / gu_s / 1e9
        roof = {"bound": "hbm", "kernel": "gemm_gate_up", "achieved": achieved, "peak": hbm,
                "unit": "GB/s", "frac": achieved / hbm, "traffic": traffic_for(wl),
                "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)" if src == "measured" else src,
                "algorithmic_bytes_per_launch": alg["gate_up_bytes"],
                "us_per_launch": per_kernel_us[gu]}
    res = {
        "workload": workload_desc(wl), "tokens_per_step": T, "steps": steps,
        "us_per_layer": ms * 1000.0, "value": T / (ms / 1000.0), "unit": UNIT,
        "touched_experts": alg["touched_experts"],
        "expert_loads": {"max": int(counts.max()), "empty": int((counts == 0).sum())},
        "roofline": roof,
        "layer_roofline": {"bytes": alg["layer_bytes"], "flops": alg["layer_flops"],
                           "t_roof_us": t_roof * 1e6, "frac": t_roof / (ms / 1000.0),
                           "basis": f"max(bytes / {hbm} GB/s, flops / {bf16_sus} TF/s) ({src}); "
                                    f"against the nominal 8 TB/s / 2.25 PF: "
                                    f"{max(alg['layer_bytes'] / 8e12, alg['layer_flops'] / 2.25e15) / (ms / 1000.0):.3f}"},
        "kernels_us": {n: round(float(v), 3) for n, v in zip(names, per_kernel_us)},
        "kernels_note": "separate pass with an event between kernels (no overlap between them)",
        "clocks": clk,
        "gpu_launches": launches_per_forward(wl, len(names)) * steps,
        "ms_per_step": ms,
    }
    return res, blk, fwd


# The configurations of the specification measured beside the headline in
# the default run: the 4-bit canvas, the Zipf-skewed batch of 8 canvases and
# one layer of the 30-layer 4-bit stack at its 16 384 tokens.
EXTRA_CONFIGS = ("canvas256_q4", "batch2048_zipf", "stack30_q4_layer")


def extra_config(name, dev, steps, warmup):
    import moe_inputs as mi
    if name == "stack30_q4_layer":
        wl = mi.get_workload("stack30_q4")
        p = mi.make_layer_inputs(wl, layer=0)
        h_np = mi.make_tokens(wl)
        res, blk, _ = measure_layer(wl, p, h_np, dev, steps, warmup, budget_s=2.0)
        res["workload"] = ("stack30_q4 layer 0 (one layer of the 30-layer stack, its own "
                           "weights and layer scalar): " + workload_desc(wl))
    else:
        wl = mi.get_workload(name)
        p = mi.make_layer_inputs(wl)
        res, blk, _ = measure_layer(wl, p, mi.make_tokens(wl), dev, steps, warmup, budget_s=2.0)
    blk.close()
    return res


def run_ours(args):
    import torch

    import moe_expert_ffn_dg_gb300 as pkg
    import moe_inputs as mi
    from moe_expert_ffn_dg_gb300 import replicas

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pkg.build()
    pkg.load_library()

    wl = mi.get_workload(args.workload)
    if args.tokens:
        wl = mi.get_workload(args.workload, tokens=args.tokens)
    p = mi.make_layer_inputs(wl)
    # each replica processes its own canvas (data parallel over canvases)
    h_np = mi.make_tokens(mi.get_workload(args.workload, seed=replicas.replica_seed(wl.seed, rank),
                                          tokens=wl.tokens))
    res, blk, fwd = measure_layer(wl, p, h_np, dev, args.steps, args.warmup, local,
                                  neighbours=args.neighbours, dist=dist)

    # end to end through the host-buffer entry point: H2D of h, forward,
    # D2H of the output, stream synchronised every step
    h_host = torch.from_numpy(h_np.view(np.int16)).view(torch.bfloat16).pin_memory()
    o_host = torch.empty_like(h_host).pin_memory()
    for _ in range(3):
        blk.forward_host(h_host, o_host, 1.0)
    e2e_steps = max(10, min(args.steps, 2000))
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        blk.forward_host(h_host, o_host, 1.0)
    e2e_s = time.perf_counter() - t0
    blk.close()

    ms = res["ms_per_step"]
    value = replicas.aggregate_throughput(world, wl.tokens, ms / 1000.0)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": res["workload"] + (
                       "; fused with the decoder layer's neighbours (post-attention residual "
                       "norm in, next layer's input norm out)" if args.neighbours else ""),
                   "tokens_per_step": wl.tokens,
                   "us_per_layer": ms * 1000.0, "parallelism": f"replicas x{world}",
                   "weights": "bf16" if not wl.quant else ("NVFP4 experts and dense" if wl.quant[0] == 16 else f"u{wl.quant[0]} g64 affine experts, u{wl.quant[1]} dense") + f", u{wl.quant[2]} router, decoded to bf16 on chip",
                   "l2": f"no flush: {res['layer_roofline']['bytes'] / 1e9:.3f} GB of weights per "
                         f"step, {res['layer_roofline']['bytes'] / 129e6:.1f}x the 129 MB L2",
                   "touched_experts": res["touched_experts"],
                   "timing": "value and ms_per_step from an event-free pass; kernels_us from a "
                             "separate pass"},
        "roofline": res["roofline"],
        "layer_roofline": res["layer_roofline"],
        "kernels_us": res["kernels_us"],
        "e2e": {"value": world * wl.tokens * e2e_steps / e2e_s, "unit": UNIT,
                "h2d_bytes_per_step": int(h_host.numel() * 2),
                "d2h_bytes_per_step": int(o_host.numel() * 2), "steps": e2e_steps,
                **({"note": "the plain block through the host-buffer entry point"}
                   if args.neighbours else {})},
        "clocks": res["clocks"],
        "gpu_launches": res["gpu_launches"],
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, p, h_np)
    # the other configurations, one GPU, in the same process (rank 0 of a
    # single-GPU run only)
    if world == 1 and not args.no_extra and args.workload == WORKLOAD and not args.tokens \
            and not args.neighbours:
        line["extra_configs"] = {n: extra_config(n, dev, args.steps, args.warmup)
                                 for n in EXTRA_CONFIGS}
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="time the headline configuration only")
    ap.add_argument("--tokens", type=int, default=0,
                    help="token count of a one-layer workload (default: the workload's own)")
    ap.add_argument("--neighbours", action="store_true",
                    help="time the block fused with the decoder layer's neighbouring norms")
    ap.add_argument("--workload", default=WORKLOAD,
                    choices=["canvas256", "canvas256_q4", "canvas256_q4d8", "canvas256_fp4",
                             "batch2048_zipf",
                             "stack30_q4", "sc_canvas256", "sc_canvas256_q4",
                             "sc_canvas256_q8"])
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "stack30_q4":
        run_stack(args)
    elif args.workload.startswith("sc_"):
        run_sc(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
