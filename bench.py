"""Benchmark: one GPT-MLP block forward + backward through the NVFP4 / MXFP8 hot path.

Workload (the configuration that passes through every step of the path): tokens 16384,
d_model 4096, ffn 16384; X ~ N(0,1) with 0.1% outliers x50, W1/W2 ~ N(0,0.02),
dY ~ Student-t(3) * 1e-3, all bf16 and synthetic. One step = 1D quantize of X and of
GELU(H), 16x16 quantize of W1 and W2, two NVFP4 GEMMs forward (GELU and max|GELU| in the
first one's epilogue); four MXFP8 requants with stochastic rounding (two with the 16-point
RHT) and two MXFP8 GEMMs per layer backward (GELU' in the second layer's dgrad epilogue).
The metric is the step's dense GEMM throughput (6 x 2 M D F FLOPs per step) in TFLOP/s.
The line also reports the same step with the activations quantized per token row with
Four Over Six block scales ("per_token_4over6"), timed separately, the MoE combine wire
format (RHT32 + S2F6) at the MoE layer's size ("combine_codec"), and MXFP4 beside NVFP4 on the
weight sweep's largest shape ("mxfp4_vs_nvfp4").

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torchrun, one process per GPU, each an independent replica of the
step on its own batch (weak scaling; the path needs no collective). The reference arm
times the CPU oracle on a bounded sample of the same step and extrapolates.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "NVFP4 GEMM TFLOPS & quantize GB/s at 1 GB300, % of FP4 peak / HBM roofline"
WORKLOAD = "gpt_mlp_fwd_bwd_16384x4096x16384"
M_TOK, D_MODEL, F_FFN = 16384, 4096, 16384
SEED = 4                     # configuration index of this workload

# nominal dense tensor-core ratios to bf16 (NVFP4 13.5 / MXFP8 4.5 / bf16 2.25 PFLOP/s)
RATIO_FP8, RATIO_FP4 = 2.0, 6.0
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# algorithmic bytes per element of the HBM-bound calls. A quantize call is two kernels, the
# per-tensor amax pass (reads 2 B) and the quantize pass (reads 2 B, writes codes + scales),
# and is timed as one call, so its bytes include both passes.
BYTES_PER_ELEM = {
    "quantize_1d": 2.0 + 2.0 + 0.5 + 1 / 16,
    "quantize_1d_given_amax": 2.0 + 0.5 + 1 / 16,
    "quantize_2d": 2.0 + 2.0 + 0.5 + 1 / 256,
    "requant_bf16": 2.0 + 1 + 1 / 32,
    "requant_nvfp4_1d": 0.5 + 1 / 16 + 1 + 1 / 32,
    "requant_nvfp4_2d": 0.5 + 1 / 256 + 1 + 1 / 32,
    # per-token form: one pass, no amax kernel (the 4-byte row scale is left out: < 0.1%)
    "quantize_1d_rows46": 2.0 + 0.5 + 1 / 16,
    # combine wire format (RHT32 + S2F6, 8.25 bits per value)
    "combine_encode_f32": 4.0 + 1 + 1 / 32,
    "combine_encode_bf16": 2.0 + 1 + 1 / 32,
    "combine_decode_k1_f32": 1 + 1 / 32 + 4.0,
    "combine_decode_k2_bf16": 2 * (1 + 1 / 32) + 2.0,
    # MXFP4 (one pass: E8M0 per 32 needs no tensor amax)
    "quantize_mxfp4": 2.0 + 0.5 + 1 / 32,
    "quantize_mxfp4_rht32": 2.0 + 0.5 + 1 / 32,
}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK), "fallback"


def ncu_traffic(kind):
    """DRAM bytes per launch of `kind` from the committed ncu summary, or None when any of
    the kernel's sources changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kind)
    except (OSError, ValueError):
        return None
    if not rec:
        return None
    h = hashlib.sha256()
    for name in rec["sources"]:
        src = os.path.join(ROOT, "mxfp8_precision_numerics_gb300", "csrc", name)
        if not os.path.exists(src):
            return None
        with open(src, "rb") as f:
            h.update(f.read())
    if h.hexdigest()[:16] != rec["source_sha"]:
        return None
    return rec["dram_bytes_per_launch"]


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.tmp = None

    def __enter__(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.tmp, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.tmp is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.tmp.flush()
        with open(self.tmp.name) as f:
            rows = [r.strip().split(", ") for r in f if r.strip()]
        os.unlink(self.tmp.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for name, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------- our arm
def make_inputs(seed):
    from mxfp8_precision_numerics_gb300 import inputs as I
    x = I.normal_with_outliers(M_TOK, D_MODEL, seed=seed)
    w1 = I.normal(F_FFN, D_MODEL, seed=seed * 10 + 1, std=0.02)
    w2 = I.normal(D_MODEL, F_FFN, seed=seed * 10 + 2, std=0.02)
    dy = I.student_t(M_TOK, D_MODEL, seed=seed * 10 + 3)
    return x, w1, w2, dy, I.sr_seed(seed), I.rht_signs(seed)


class EventLog:
    """CUDA events around each library call of a step, on the launching stream."""

    def __init__(self, torch):
        self.torch = torch
        self.marks = []          # (kind, units, start event, end event)
        self.on = False

    def wrap(self, kind, units, fn, *a, **k):
        if not self.on:
            return fn(*a, **k)
        s = self.torch.cuda.Event(enable_timing=True)
        e = self.torch.cuda.Event(enable_timing=True)
        s.record()
        out = fn(*a, **k)
        e.record()
        self.marks.append((kind, units, s, e))
        return out

    def totals(self):
        agg = {}
        for kind, units, s, e in self.marks:
            ms = s.elapsed_time(e)
            t = agg.setdefault(kind, [0, 0.0, 0.0])
            t[0] += 1
            t[1] += ms
            t[2] += units
        return agg


def mlp_step(F, torch, ins, log, seed, signs, outer="tensor"):
    """One forward + backward of the MLP block, every call logged by kind. outer="row": the
    activations (X and GELU(H)) take one outer scale per token row and 4/6 block scales."""
    x, w1, w2, dy = ins
    M, D, Fh = M_TOK, D_MODEL, F_FFN
    L = log.wrap
    rows = outer == "row"
    x_kind = F.IN_NVFP4_1D_ROWS if rows else F.IN_NVFP4_1D
    # ---- forward
    if rows:
        xc, xs, xsd = L("quantize_1d_rows46", M * D, F.quantize_1d_rows, x, True)
    else:
        xc, xs, xsd, _ = L("quantize_1d", M * D, F.quantize_1d, x)
    w1c, w1s, w1d, _ = L("quantize_2d", Fh * D, F.quantize_2d, w1)
    # layer 1 with GELU in its epilogue: h, a = GELU(h) and max|a| (layer 2's quantize amax)
    if rows:
        h, a = L("gemm_nvfp4", 2.0 * M * Fh * D, F.gemm_nvfp4_gelu_rows, xc, xs, xsd, w1c, w1s, F.SCALE_2D, w1d)
        ac, as_, ad = L("quantize_1d_rows46", M * Fh, F.quantize_1d_rows, a, True)
    else:
        h, a, a_amax = L("gemm_nvfp4", 2.0 * M * Fh * D, F.gemm_nvfp4_gelu, xc, xs, xsd, w1c, w1s, F.SCALE_2D, w1d)
        ac, as_, ad, _ = L("quantize_1d_given_amax", M * Fh, F.quantize_1d, a, amax_in=a_amax)
    w2c, w2s, w2d, _ = L("quantize_2d", D * Fh, F.quantize_2d, w2)
    gemm2 = F.gemm_nvfp4_rows if rows else F.gemm_nvfp4
    y = L("gemm_nvfp4", 2.0 * M * D * Fh, gemm2, ac, as_, ad, w2c, w2s, F.SCALE_2D, w2d, torch.bfloat16)
    # ---- backward, layer 2: dA = dY W2, dW2 = dY^T A_q
    g = L("requant_bf16", M * D, F.requant_mxfp8, F.IN_BF16, dy, None, None, M, D, 0, 0, 0, F.SR, seed, F.TAG_DY_ROWS)
    w2t = L("requant_nvfp4_2d", D * Fh, F.requant_mxfp8, F.IN_NVFP4_2D, w2c, w2s, w2d, D, Fh, 1, 0, 0, F.SR, seed, F.TAG_WT)
    # layer 2's dgrad with GELU' in its epilogue: dh = (dY W2) * GELU'(h)
    dh = L("gemm_mxfp8", 2.0 * M * Fh * D, F.gemm_mxfp8_dgelu, g[0], g[1], w2t[0], w2t[1], h)
    gt = L("requant_bf16", M * D, F.requant_mxfp8, F.IN_BF16, dy, None, None, M, D, 1, 1, signs, F.SR, seed, F.TAG_DY_T)
    at = L("requant_nvfp4_1d", M * Fh, F.requant_mxfp8, x_kind, ac, as_, ad, M, Fh, 1, 1, signs, F.SR, seed, F.TAG_XT)
    dw2 = L("gemm_mxfp8", 2.0 * D * Fh * M, F.gemm_mxfp8, gt[0], gt[1], at[0], at[1], torch.float32)
    # ---- backward, layer 1: dX = dH W1, dW1 = dH^T X_q  (own counter stream: seed2)
    seed2 = seed ^ 0x9E3779B97F4A7C15
    g1 = L("requant_bf16", M * Fh, F.requant_mxfp8, F.IN_BF16, dh, None, None, M, Fh, 0, 0, 0, F.SR, seed2, F.TAG_DY_ROWS)
    w1t = L("requant_nvfp4_2d", Fh * D, F.requant_mxfp8, F.IN_NVFP4_2D, w1c, w1s, w1d, Fh, D, 1, 0, 0, F.SR, seed2, F.TAG_WT)
    dx = L("gemm_mxfp8", 2.0 * M * D * Fh, F.gemm_mxfp8, g1[0], g1[1], w1t[0], w1t[1], torch.bfloat16)
    g1t = L("requant_bf16", M * Fh, F.requant_mxfp8, F.IN_BF16, dh, None, None, M, Fh, 1, 1, signs, F.SR, seed2, F.TAG_DY_T)
    xt = L("requant_nvfp4_1d", M * D, F.requant_mxfp8, x_kind, xc, xs, xsd, M, D, 1, 1, signs, F.SR, seed2, F.TAG_XT)
    dw1 = L("gemm_mxfp8", 2.0 * Fh * D * M, F.gemm_mxfp8, g1t[0], g1t[1], xt[0], xt[1], torch.float32)
    return y, dx, dw1, dw2


LAUNCHES_PER_STEP = {
    "amax": 3, "quantize_1d": 2, "quantize_2d": 2, "gemm_nvfp4": 2, "requant": 8, "gemm_mxfp8": 4,
}
# per-token form: the weights' two amax passes, no activation amax
LAUNCHES_PER_STEP_ROWS = {
    "amax": 2, "quantize_1d_rows": 2, "quantize_2d": 2, "gemm_nvfp4": 2, "requant": 8, "gemm_mxfp8": 4,
}
STEP_FLOPS = 6 * 2.0 * M_TOK * D_MODEL * F_FFN


def summarize_kernels(kinds, peaks):
    """Per call kind: launches, average duration and achieved rate against its roofline."""
    kernels = {}
    for kind, (n, tot_ms, units) in sorted(kinds.items()):
        avg = tot_ms / n
        if kind.startswith("gemm"):
            tf = units / (tot_ms * 1e-3) / 1e12
            fp4 = kind.startswith(("gemm_nvfp4", "gemm_mxfp4"))
            peak = peaks["bf16_tflops_sustained"] * (RATIO_FP4 if fp4 else RATIO_FP8)
            kernels[kind] = {"launches": n, "avg_ms": round(avg, 4), "achieved": round(tf, 1),
                             "unit": "TFLOP/s", "peak": round(peak, 1), "frac": round(tf / peak, 4)}
        else:
            gbs = units * BYTES_PER_ELEM[kind] / (tot_ms * 1e-3) / 1e9
            two_pass = kind in ("quantize_1d", "quantize_2d")
            kernels[kind] = {"launches": n, "avg_ms": round(avg, 4), "achieved": round(gbs, 1),
                             "unit": "GB/s (amax + quantize passes)" if two_pass else "GB/s",
                             "peak": peaks["hbm_gbs"], "frac": round(gbs / peaks["hbm_gbs"], 4)}
        kernels[kind]["traffic"] = ncu_traffic(kind)      # DRAM bytes per launch (ncu), or None
    return kernels


def combine_section(F, torch, dev, peaks, iters=10):
    """The MoE combine wire format (RHT32 + S2F6) at the MoE layer's size: the expert down
    projection as a grouped NVFP4 GEMM with a bf16 output and with the encode in its epilogue,
    the stand-alone encoder, and the receiver's decode (one and two arrivals per token)."""
    from mxfp8_precision_numerics_gb300 import inputs as I
    T, D, FE, E = 8192, 4096, 1536, 8          # tokens, d_model, expert ffn, experts (top-1, 1024 each)
    signs = 0x9E3779B9
    h = I.normal(T, FE, seed=31).to(dev)
    w2 = I.normal(E * D, FE, seed=32, std=0.02).view(E, D, FE).to(dev)
    hc, hs, hsd, _ = F.quantize_1d(h)
    wc, ws, wsd, _ = F.quantize_2d(w2)
    offs = [i * (T // E) for i in range(E + 1)]
    y32 = I.student_t(T, D, seed=33, df=3, scale=1.0).float().to(dev)
    y16 = y32.to(torch.bfloat16)
    codes2, e82 = F.combine_encode(I.student_t(2 * T, D, seed=34, df=3, scale=1.0).float().to(dev), signs)
    log = EventLog(torch)
    L = log.wrap
    flops = 2.0 * T * D * FE

    def once():
        L("gemm_nvfp4_grouped_bf16", flops, F.gemm_nvfp4, hc, hs, hsd, wc, ws, F.SCALE_2D, wsd, torch.bfloat16,
          E, offs)
        c, e8 = L("gemm_nvfp4_grouped_combine", flops, F.gemm_nvfp4_combine, hc, hs, hsd, wc, ws, F.SCALE_2D, wsd,
                  signs, E, offs)
        L("combine_encode_f32", T * D, F.combine_encode, y32, signs)
        L("combine_encode_bf16", T * D, F.combine_encode, y16, signs)
        L("combine_decode_k1_f32", T * D, F.combine_decode, c, e8, 1, signs, torch.float32)
        L("combine_decode_k2_bf16", T * D, F.combine_decode, codes2, e82, 2, signs, torch.bfloat16)

    for _ in range(3):
        once()
    torch.cuda.synchronize()
    log.on = True
    for _ in range(iters):
        once()
    torch.cuda.synchronize()
    log.on = False
    st = F.fp4q_device_status()
    if st != F.OK:
        raise RuntimeError("device status after the combine section: " + F.status_str(st))
    return {"workload": f"MoE combine: {T} tokens x d_model {D}, {E} experts x {T // E} tokens (top-1), "
                        f"expert ffn {FE}; decode k=2 on {2 * T} arrivals; inputs N(0,1) / Student-t(3)",
            "iterations": iters, "kernels": summarize_kernels(log.totals(), peaks)}


def format_section(F, torch, dev, peaks, iters=10):
    """MXFP4 beside NVFP4 on the weight sweep's largest shape (X 16384 x 4096, W 14336 x 4096):
    the activation quantizers and the bf16-output GEMMs."""
    from mxfp8_precision_numerics_gb300 import inputs as I
    M, N, K = 16384, 14336, 4096
    signs = 0x5EED1234
    x = I.normal_with_outliers(M, K, seed=3).to(dev)
    w = I.normal(N, K, seed=30, std=0.02).to(dev)
    xc, xs, xsd, _ = F.quantize_1d(x)
    wc, ws, wsd, _ = F.quantize_2d(w)
    mxc, mxe = F.quantize_mxfp4(x)
    mwc, mwe = F.quantize_mxfp4(w)
    log = EventLog(torch)
    L = log.wrap
    flops = 2.0 * M * N * K

    def once():
        L("quantize_1d", M * K, F.quantize_1d, x)
        L("quantize_mxfp4", M * K, F.quantize_mxfp4, x)
        L("quantize_mxfp4_rht32", M * K, F.quantize_mxfp4, x, True, signs)
        L("gemm_nvfp4_w2d", flops, F.gemm_nvfp4, xc, xs, xsd, wc, ws, F.SCALE_2D, wsd, torch.bfloat16)
        L("gemm_mxfp4", flops, F.gemm_mxfp4, mxc, mxe, mwc, mwe, torch.bfloat16)

    for _ in range(3):
        once()
    torch.cuda.synchronize()
    log.on = True
    for _ in range(iters):
        once()
    torch.cuda.synchronize()
    log.on = False
    st = F.fp4q_device_status()
    if st != F.OK:
        raise RuntimeError("device status after the format section: " + F.status_str(st))
    return {"workload": f"X {M}x{K} N(0,1)+0.1% x50, W {N}x{K} N(0,0.02); bf16 GEMM outputs",
            "iterations": iters, "kernels": summarize_kernels(log.totals(), peaks)}


def max_over_ranks(values, device):
    """Element-wise max of per-rank timings (the slowest rank sets the job time)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def run_ours(args, rank, world, local_rank):
    import torch
    from mxfp8_precision_numerics_gb300 import fp4q as F

    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    x, w1, w2, dy, seed, signs = make_inputs(SEED + 100 * rank)
    host = [t.pin_memory() for t in (x, w1, w2, dy)]
    ins = [t.to(dev) for t in host]
    torch.cuda.synchronize()
    log = EventLog(torch)

    def barrier():
        if dist is not None:
            dist.barrier()

    for _ in range(args.warmup):
        mlp_step(F, torch, ins, log, seed, signs)
    torch.cuda.synchronize()
    st = F.fp4q_device_status()
    if st != F.OK:
        raise RuntimeError("device status after warm-up: " + F.status_str(st))

    # ---- timed region: inputs resident in HBM (working set >> L2: no flush needed)
    log.on = True
    props = torch.cuda.get_device_properties(dev)
    smi_id = ("GPU-" + str(props.uuid)) if getattr(props, "uuid", None) else str(local_rank)
    with ClockSampler(smi_id) as clk:
        barrier()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(args.steps):
            mlp_step(F, torch, ins, log, seed, signs)
        t1.record()
        torch.cuda.synchronize()
        barrier()
    log.on = False
    ms = t0.elapsed_time(t1)
    clocks = clk.summary()
    kinds = log.totals()

    # ---- end to end through the public API with host buffers (pinned)
    # Every step copies its inputs in from pinned host memory and its results (Y, dX, dW1, dW2)
    # back out, as a training loop feeding the layer from the host would: one copy stream brings
    # step i+1's inputs in while step i computes, another takes step i's results out as they are
    # done (the two directions use separate copy engines and run at the same time). Device
    # buffers and pinned result buffers are allocated before the timed loop. The device events
    # and the host wall clock bracket the loop.
    e2e_steps = max(1, args.steps // 2)
    copy = torch.cuda.Stream(device=dev)          # host -> device
    copy_out = torch.cuda.Stream(device=dev)      # device -> host
    comp = torch.cuda.current_stream(dev)
    dbuf = [[torch.empty_like(t, device=dev) for t in host] for _ in range(2)]
    outs_host = None
    h2d = sum(t.numel() * t.element_size() for t in host)
    d2h = 0

    def e2e_loop(nsteps):
        nonlocal outs_host, d2h
        in_ready = [torch.cuda.Event() for _ in range(2)]
        buf_free = [torch.cuda.Event() for _ in range(2)]
        out_done = torch.cuda.Event()
        with torch.cuda.stream(copy):
            for d, hsrc in zip(dbuf[0], host):
                d.copy_(hsrc, non_blocking=True)
            in_ready[0].record(copy)
        for i in range(nsteps):
            b = i % 2
            comp.wait_event(in_ready[b])
            outs = mlp_step(F, torch, dbuf[b], log, seed, signs)
            buf_free[b].record(comp)
            out_done.record(comp)
            if i + 1 < nsteps:
                with torch.cuda.stream(copy):
                    nb = (i + 1) % 2
                    if i >= 1:
                        copy.wait_event(buf_free[nb])
                    for d, hsrc in zip(dbuf[nb], host):
                        d.copy_(hsrc, non_blocking=True)
                    in_ready[nb].record(copy)
            with torch.cuda.stream(copy_out):
                copy_out.wait_event(out_done)
                if outs_host is None:
                    outs_host = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
                for oh, o in zip(outs_host, outs):
                    o.record_stream(copy_out)
                    oh.copy_(o, non_blocking=True)
            d2h = sum(o.numel() * o.element_size() for o in outs)
        comp.wait_stream(copy)
        comp.wait_stream(copy_out)

    e2e_loop(2)                      # warm-up: allocations and first-touch outside the timing
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    e0.record(comp)
    e2e_loop(e2e_steps)
    e1.record(comp)
    torch.cuda.synchronize()
    wall1 = time.perf_counter()
    barrier()
    e2e_event_ms, e2e_wall_ms = e0.elapsed_time(e1) / e2e_steps, (wall1 - wall0) * 1e3 / e2e_steps
    e2e_ms = max(e2e_event_ms, e2e_wall_ms)
    st = F.fp4q_device_status()
    if st != F.OK:
        raise RuntimeError("device status after timing: " + F.status_str(st))

    # ---- the same step with per-token activation scales and 4/6 block scales
    # (4bit.vizuara.ai §10), timed on its own after warm-up
    rlog = EventLog(torch)
    for _ in range(3):
        mlp_step(F, torch, ins, rlog, seed, signs, outer="row")
    r_steps = max(2, args.steps // 4)
    barrier()
    torch.cuda.synchronize()
    rlog.on = True
    r0 = torch.cuda.Event(enable_timing=True)
    r1 = torch.cuda.Event(enable_timing=True)
    r0.record()
    for _ in range(r_steps):
        mlp_step(F, torch, ins, rlog, seed, signs, outer="row")
    r1.record()
    torch.cuda.synchronize()
    barrier()
    rlog.on = False
    r_ms = r0.elapsed_time(r1) / r_steps
    st = F.fp4q_device_status()
    if st != F.OK:
        raise RuntimeError("device status after the per-token step: " + F.status_str(st))

    # ---- max over ranks
    per_step, e2e_ms, r_ms = max_over_ranks([ms / args.steps, e2e_ms, r_ms], dev)
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return None

    peaks, peak_src = load_peaks()
    kernels = summarize_kernels(kinds, peaks)
    dom = max(kinds.items(), key=lambda kv: kv[1][1])[0]
    n, tot_ms, units = kinds[dom]
    traffic = ncu_traffic(dom)
    if dom.startswith("gemm"):
        roof = {"kernel": dom, "bound": "tensor", "achieved": kernels[dom]["achieved"], "peak": kernels[dom]["peak"],
                "unit": "TFLOP/s", "frac": kernels[dom]["frac"], "traffic": traffic,
                "peak_source": f"{peak_src} bf16 sustained x {RATIO_FP4 if dom == 'gemm_nvfp4' else RATIO_FP8:g} (nominal dtype ratio)",
                "algorithmic_per_launch": f"{units / n:.4g} FLOP"}
    else:
        roof = {"kernel": dom, "bound": "hbm", "achieved": kernels[dom]["achieved"], "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": kernels[dom]["frac"], "traffic": traffic, "peak_source": peak_src}
    value = STEP_FLOPS / (per_step * 1e-3) / 1e12
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4(e2m1,e4m3 scale)/mxfp8(e4m3,e8m0) x fp32-accum",
        "data": "synthetic (seeded bf16: X N(0,1)+0.1% x50 outliers, W N(0,0.02), dY Student-t(3)*1e-3)",
        "config": {"workload": WORKLOAD, "tokens": M_TOK, "d_model": D_MODEL, "ffn": F_FFN,
                   "step": "MLP block fwd (2 NVFP4 GEMMs) + bwd (4 MXFP8 GEMMs, SR, RHT16 on wgrad)",
                   "l2": "no flush: per-step working set > 4 GB >> 129 MB L2", "parallelism": f"replicas x{world}"},
        "roofline": roof,
        "kernels": kernels,
        "e2e": {"value": round(STEP_FLOPS / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": round(e2e_ms, 3), "event_ms": round(e2e_event_ms, 3),
                "wall_ms": round(e2e_wall_ms, 3)},
        "gpu_launches": int(sum(LAUNCHES_PER_STEP.values()) * args.steps),
        "clocks": clocks,
        "per_token_4over6": {
            "what": "the same step with the activations quantized per token row with 4/6 block scales "
                    "(one pass, no activation amax), per-row outer scales through both GEMM epilogues "
                    "and the X^T requantizations",
            "value": round(STEP_FLOPS / (r_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "ms_per_step": round(r_ms, 4), "steps": r_steps, "warmup": 3,
            "gpu_launches": int(sum(LAUNCHES_PER_STEP_ROWS.values()) * r_steps),
            "kernels": summarize_kernels(rlog.totals(), peaks),
        },
    }
    res["combine_codec"] = combine_section(F, torch, dev, peaks)
    res["mxfp4_vs_nvfp4"] = format_section(F, torch, dev, peaks)
    if world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(args.cpu_sample)
    if dist is not None:
        dist.destroy_process_group()
    return res


# ---------------------------------------------------------------------------- CPU oracle
def _oracle_sample_worker(frac_rows):
    """Time the CPU oracle on a bounded sample of one step and extrapolate to the full
    step. Runs in a fresh single-threaded process (spawned, never forked after CUDA)."""
    import numpy as np
    import oracle as O
    from mxfp8_precision_numerics_gb300 import inputs as I

    M, D, Fh = M_TOK, D_MODEL, F_FFN
    r = max(16, int(frac_rows))
    seed, signs = I.sr_seed(SEED), I.rht_signs(SEED)
    xs = I.bf16_bits(I.normal_with_outliers(r, D, seed=SEED))
    w1s = I.bf16_bits(I.normal(r, D, seed=41, std=0.02))
    w2s = I.bf16_bits(I.normal(r, Fh, seed=42, std=0.02))
    hs = I.bf16_bits(I.normal(r, Fh, seed=43))
    dys = I.bf16_bits(I.student_t(r, D, seed=44))
    dhs = I.bf16_bits(I.student_t(r, Fh, seed=45))
    est = 0.0

    def timed(fn):
        t = time.perf_counter()
        out = fn()
        return out, time.perf_counter() - t

    # forward quantizes: rows scale linearly
    (xc, xsc, _, xsd), t = timed(lambda: O.quantize_1d(xs)); est += t * M / r
    (w1c, w1t, _, w1d), t = timed(lambda: O.quantize_2d(w1s)); est += t * Fh / r
    (ac, asc, _, ad), t = timed(lambda: O.quantize_1d(hs)); est += t * M / r
    (w2c, w2t, _, w2d), t = timed(lambda: O.quantize_2d(w2s)); est += t * D / r

    def gemm_time(deq_a, rows_a_full, deq_b, rows_b_full):
        A, ta = timed(deq_a)
        B, tb = timed(deq_b)
        _, tm = timed(lambda: A @ B.T)
        return ta * rows_a_full / A.shape[0] + tb * rows_b_full / B.shape[0] + \
            tm * (rows_a_full / A.shape[0]) * (rows_b_full / B.shape[0])

    est += gemm_time(lambda: O.dequant_nvfp4(xc, xsc, 1, xsd), M, lambda: O.dequant_nvfp4(w1c, w1t, 2, w1d), Fh)
    est += gemm_time(lambda: O.dequant_nvfp4(ac, asc, 1, ad), M, lambda: O.dequant_nvfp4(w2c, w2t, 2, w2d), D)
    # backward requants: 16 output rows of each; (kind, data, scales, s_dec, sample rows, cols,
    # transpose, rht, full output rows, full output cols)
    out_r = 16
    for kind, data, sc, sd, rows, cols, tr, rht, f_or, f_oc in (
            (O.IN_BF16, dys, None, 1.0, r, D, False, False, M, D),          # dY rows
            (O.IN_NVFP4_2D, w2c, w2t, w2d, r, Fh, True, False, Fh, D),      # W2^T
            (O.IN_BF16, dys, None, 1.0, r, D, True, True, D, M),            # dY^T
            (O.IN_NVFP4_1D, ac, asc, ad, r, Fh, True, True, Fh, M),         # A_q^T
            (O.IN_BF16, dhs, None, 1.0, r, Fh, False, False, M, Fh),        # dH rows
            (O.IN_NVFP4_2D, w1c, w1t, w1d, r, D, True, False, D, Fh),       # W1^T
            (O.IN_BF16, dhs, None, 1.0, r, Fh, True, True, Fh, M),          # dH^T
            (O.IN_NVFP4_1D, xc, xsc, xsd, r, D, True, True, D, M)):         # X_q^T
        n_out = min(out_r, cols if tr else rows)
        _, t = timed(lambda: O.requant_mxfp8(kind, data, sc, sd, rows, cols, tr, rht, signs, O.SR, seed, 1,
                                             out_rows=(0, n_out)))
        sample_elems = n_out * (rows if tr else cols)
        est += t * (f_or * f_oc) / sample_elems
    # MXFP8 GEMMs: dequant + product of sampled rows, extrapolated
    e4 = np.random.default_rng(0).integers(0, 0x7E, (r, Fh), dtype=np.uint8)
    e8 = np.full((r, Fh // 32), 127, np.uint8)
    for rows_a, rows_b, k in ((M, Fh, D), (D, Fh, M), (M, D, Fh), (Fh, D, M)):
        kk = min(k, Fh)
        deq = lambda: O.dequant_mxfp8(e4[:, :kk], e8[:, :kk // 32])
        t_one = gemm_time(deq, rows_a, deq, rows_b)
        est += t_one * (k / kk)
    return est


def _spawn_oracle(sample_rows, repeat):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    t = time.perf_counter()
    out = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-worker", str(sample_rows),
                          "--oracle-repeat", str(repeat)], env=env, capture_output=True, text=True, timeout=1800)
    wall = time.perf_counter() - t
    if out.returncode != 0:
        tail = out.stderr.strip().splitlines()[-1] if out.stderr.strip() else "no output"
        raise RuntimeError("oracle worker failed: " + tail)
    return json.loads(out.stdout.strip().splitlines()[-1]), wall


def cpu_baseline(sample_rows):
    """Spawn a single-threaded oracle process and time a bounded sample of one step."""
    try:
        ests, wall = _spawn_oracle(sample_rows, 1)
    except (RuntimeError, subprocess.TimeoutExpired) as e:
        return {"value": None, "unit": "TFLOP/s", "cores": 1, "kind": "oracle", "sample": str(e)}
    est_s = ests[0]
    return {"value": round(STEP_FLOPS / est_s / 1e12, 6), "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "sample": (f"{sample_rows} rows of every operand of one step (quantize; requant of 16 output rows; "
                       f"GEMM dequant + float64 product of sampled rows), extrapolated linearly to the full "
                       f"step; {wall:.1f} s wall incl. start-up; estimated full step {est_s:.0f} s"),
            "est_step_s": round(est_s, 2), "sample_wall_s": round(wall, 2)}


def run_reference(args, rank):
    """The reference arm: the CPU oracle on a bounded sample of the same step, per step."""
    if rank != 0:
        return None
    rows = max(16, args.cpu_sample // 4)
    ests, wall = _spawn_oracle(rows, args.warmup + args.steps)
    est = statistics.median(ests[args.warmup:])
    value = STEP_FLOPS / est / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(est * 1e3, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64/f32 (CPU oracle)",
        "data": "synthetic (same seeded generators)",
        "config": {"workload": WORKLOAD, "tokens": M_TOK, "d_model": D_MODEL, "ffn": F_FFN},
        "cpu_baseline": {"kind": "oracle", "cores": 1, "value": round(value, 6),
                         "sample": (f"{rows} sampled rows per operand per step, extrapolated to the full step; "
                                    f"{args.warmup + args.steps} samples in {wall:.1f} s")},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-sample", type=int, default=512, help="rows per operand in the CPU-oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-worker", type=int, default=None, help=argparse.SUPPRESS)
    ap.add_argument("--oracle-repeat", type=int, default=1, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_worker is not None:
        print(json.dumps([_oracle_sample_worker(args.oracle_worker) for _ in range(args.oracle_repeat)]))
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus and "WORLD_SIZE" in os.environ:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    if args.impl == "reference":
        res = run_reference(args, rank)
    else:
        res = run_ours(args, rank, world, local_rank)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
