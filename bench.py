"""Benchmark: one GPT-MLP block forward + backward through the NVFP4 / MXFP8 hot path.

Workload (the configuration that passes through every step of the path): tokens 16384,
d_model 4096, ffn 16384; X ~ N(0,1) with 0.1% outliers x50, W1/W2 ~ N(0,0.02),
dY ~ Student-t(3) * 1e-3, all bf16 and synthetic. One step = 1D quantize of X and of
GELU(H), 16x16 quantize of W1 and W2, two NVFP4 GEMMs forward (GELU and max|GELU| in the
first one's epilogue); per layer backward, the four MXFP8 quantizations with stochastic rounding
(two with the 16-point RHT; the output gradient's rowwise and transposed ones from one read of it)
and two MXFP8 GEMMs (GELU' in the second layer's dgrad epilogue).
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
    # the output gradient's rowwise and transposed quantizations from one read
    "requant_bf16_dual": 2.0 + 2 * (1 + 1 / 32),
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
    """nvidia-smi clock / throttle-reason samples every 20 ms while running."""
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
                 "-lms", "20"], stdout=self.tmp, stderr=subprocess.DEVNULL)
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


class StreamTap:
    """Call hook of the end-to-end loop. Before a library call the compute stream waits for the
    host-to-device copy of each step input whose memory one of the call's tensor arguments
    overlaps (once per input); after the call an event marks its outputs ready, so that their
    device-to-host copies start while the rest of the step runs. new_event() makes an event with
    .record(stream); stream has .wait_event(event)."""

    def __init__(self, new_event, stream, inputs, ready):
        self.new_event, self.stream = new_event, stream
        self.pending = [(t.data_ptr(), t.data_ptr() + t.numel() * t.element_size(), ev)
                        for t, ev in zip(inputs, ready)]
        self.done = {}

    @staticmethod
    def _tensors(args):
        for a in args:
            if isinstance(a, (tuple, list)):
                yield from StreamTap._tensors(a)
            elif hasattr(a, "data_ptr") and hasattr(a, "element_size"):
                yield a

    def wrap(self, kind, units, fn, *a, **k):
        spans = [(t.data_ptr(), t.data_ptr() + t.numel() * t.element_size())
                 for t in self._tensors(list(a) + list(k.values()))]
        keep = []
        for lo, hi, ev in self.pending:
            if any(s0 < hi and lo < s1 for s0, s1 in spans):
                self.stream.wait_event(ev)
            else:
                keep.append((lo, hi, ev))
        self.pending = keep
        out = fn(*a, **k)
        ev = self.new_event()
        ev.record(self.stream)
        for t in self._tensors(out if isinstance(out, (tuple, list)) else [out]):
            self.done[t.data_ptr()] = ev
        return out

    def finish(self):
        """The step's remaining inputs (read by no call) are waited for all the same."""
        for _, _, ev in self.pending:
            self.stream.wait_event(ev)
        self.pending = []

    def ready(self, t):
        return self.done.get(t.data_ptr())


def mlp_step(F, torch, ins, log, seed, signs, outer="tensor"):
    """One forward + backward of the MLP block (layer.mlp_step), every call logged by kind.
    outer="row": the activations (X and GELU(H)) take one outer scale per token row and 4/6
    block scales."""
    from mxfp8_precision_numerics_gb300 import layer
    x, w1, w2, dy = ins
    S = layer.mlp_step(x, w1, w2, dy, seed, signs, outer=outer, call=log.wrap)
    return S["y"], S["dx"], S["dw1"], S["dw2"]


LAUNCHES_PER_STEP = {
    "amax": 3, "quantize_1d": 2, "quantize_2d": 2, "gemm_nvfp4": 2, "requant": 6, "gemm_mxfp8": 4,
}
# per-token form: the weights' two amax passes, no activation amax
LAUNCHES_PER_STEP_ROWS = {
    "amax": 2, "quantize_1d_rows": 2, "quantize_2d": 2, "gemm_nvfp4": 2, "requant": 6, "gemm_mxfp8": 4,
}
STEP_FLOPS = 6 * 2.0 * M_TOK * D_MODEL * F_FFN


def summarize_kernels(kinds, peaks, peak_src="measured", region_s=0.0, traffic_kinds=None):
    """Per call kind: launches, average duration and achieved rate against its roofline
    (GEMMs against the tensor peak gemm_peak picks for a timed region of region_s seconds).
    DRAM traffic comes from the committed ncu captures, which were taken at the MLP step's
    shapes (and the weight sweep's largest GEMM): traffic_kinds lists the kinds that run at
    those shapes here (None: all, the step itself); the others report null."""
    kernels = {}
    for kind, (n, tot_ms, units) in sorted(kinds.items()):
        avg = tot_ms / n
        if kind.startswith("gemm"):
            tf = units / (tot_ms * 1e-3) / 1e12
            fp4 = kind.startswith(("gemm_nvfp4", "gemm_mxfp4"))
            peak, how = gemm_peak(peaks, fp4, region_s)
            kernels[kind] = {"launches": n, "avg_ms": round(avg, 4), "achieved": round(tf, 1),
                             "unit": "TFLOP/s", "peak": round(peak, 1), "frac": round(tf / peak, 4),
                             "peak_source": f"{peak_src} {how}",
                             "algorithmic_per_launch": f"{units / n:.4g} FLOP"}
        else:
            base = kind.split("_M")[0] if "_M" in kind else kind
            bpe = BYTES_PER_ELEM[base]
            gbs = units * bpe / (tot_ms * 1e-3) / 1e9
            two_pass = base in ("quantize_1d", "quantize_2d")
            kernels[kind] = {"launches": n, "avg_ms": round(avg, 4), "achieved": round(gbs, 1),
                             "unit": "GB/s (amax + quantize passes)" if two_pass else "GB/s",
                             "peak": peaks["hbm_gbs"], "frac": round(gbs / peaks["hbm_gbs"], 4),
                             "peak_source": f"{peak_src} HBM copy",
                             "algorithmic_per_launch": f"{units / n * bpe:.4g} B"}
        # DRAM bytes per launch (ncu), or None
        kernels[kind]["traffic"] = ncu_traffic(kind) if traffic_kinds is None or kind in traffic_kinds else None
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
            "iterations": iters, "kernels": summarize_kernels(log.totals(), peaks, "measured", traffic_kinds=())}


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
            "iterations": iters,
            "kernels": summarize_kernels(log.totals(), peaks, "measured", traffic_kinds=("quantize_1d",))}


FLUSH_BYTES = 256 << 20      # written between timed iterations: twice the 129 MB L2


def gemm_peak(peaks, fp4, region_s):
    """The tensor peak a GEMM rate is divided by: the measured bf16 burst figure for a timed
    region under 2 s (a kernel timed alone), the sustained one for a longer region, times the
    nominal dtype ratio."""
    burst = region_s < 2.0
    base = peaks["bf16_tflops"] if burst else peaks["bf16_tflops_sustained"]
    ratio = RATIO_FP4 if fp4 else RATIO_FP8
    return base * ratio, f"bf16 {'burst' if burst else 'sustained'} x {ratio:g}"


def timed_calls(torch, dev, once, iters, flush=True):
    """Run once(call) 3 times untimed, then `iters` timed iterations with every library call
    bracketed by CUDA events; between iterations a 256 MB buffer is written (L2 flush)."""
    log = EventLog(torch)
    buf = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    for _ in range(3):
        once(log.wrap)
    torch.cuda.synchronize()
    log.on = True
    for _ in range(iters):
        if buf is not None:
            log.on = False
            buf.zero_()
            log.on = True
        once(log.wrap)
    torch.cuda.synchronize()
    log.on = False
    return log


def roofline_of(kernels, kind):
    k = kernels[kind]
    bound = "tensor" if kind.startswith("gemm") else "hbm"
    return {"kernel": kind, "bound": bound, "achieved": k["achieved"], "peak": k["peak"], "unit": k["unit"],
            "frac": k["frac"], "traffic": k["traffic"], "peak_source": k["peak_source"]}


def configs_section(F, torch, dev, peaks, peak_src, iters=10):
    """The four other workloads, each timed on its own (3 warm-up + `iters` iterations, L2
    flushed between iterations): per call kind its launches, average time and roofline
    fraction; the config's own figure and the roofline of its dominant call."""
    from mxfp8_precision_numerics_gb300 import inputs as I
    out = {}

    def finish(name, log, workload, value, unit, extra=None, traffic_kinds=()):
        kinds = log.totals()
        region_s = sum(t for _, t, _ in kinds.values()) * 1e-3
        kern = summarize_kernels(kinds, peaks, peak_src, region_s, traffic_kinds)
        dom = max(kinds.items(), key=lambda kv: kv[1][1])[0]
        rec = {"workload": workload, "iterations": iters, "value": value(kinds), "unit": unit,
               "kernels": kern, "roofline": roofline_of(kern, dom)}
        if extra:
            rec.update(extra(kern))
        out[name] = rec

    def per_iter_ms(kinds):
        return sum(t for _, t, _ in kinds.values()) / iters

    # ---- single NVFP4 linear forward: X 256 x 512 (+outliers), W 256 x 512, Y fp32 256 x 256
    x = I.normal_with_outliers(256, 512, seed=0).to(dev)
    w = I.normal(256, 512, seed=100, std=0.02).to(dev)

    def c1(L):
        xc, xs, xsd, _ = L("quantize_1d", 256 * 512, F.quantize_1d, x)
        wc, ws, wsd, _ = L("quantize_2d", 256 * 512, F.quantize_2d, w)
        L("gemm_nvfp4", 2.0 * 256 * 256 * 512, F.gemm_nvfp4, xc, xs, xsd, wc, ws, F.SCALE_2D, wsd, torch.float32)

    finish("linear_fwd_256x512", timed_calls(torch, dev, c1, iters),
           "X 256x512 N(0,1)+0.1% x50, W 256x512 N(0,0.02); 1D + 2D quantize, NVFP4 GEMM fp32 out",
           lambda k: round(per_iter_ms(k) * 1e3, 2), "us per forward (launch-latency bound)")
    # the same forward (5 kernels) captured once in a CUDA graph and replayed: the host's per-call
    # overhead leaves the measurement; L2 flushed before every replay
    def c1_direct():
        xc, xs, xsd, _ = F.quantize_1d(x)
        wc, ws, wsd, _ = F.quantize_2d(w)
        return F.gemm_nvfp4(xc, xs, xsd, wc, ws, F.SCALE_2D, wsd, torch.float32)

    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        for _ in range(3):
            c1_direct()
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        c1_direct()
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    times = []
    for i in range(3 + iters):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        graph.replay()
        e1.record()
        torch.cuda.synchronize()
        if i >= 3:
            times.append(e0.elapsed_time(e1))
    st = F.fp4q_device_status()
    if st != F.OK:
        raise RuntimeError("device status after the graph replays: " + F.status_str(st))
    out["linear_fwd_256x512"]["graph"] = {
        "what": "the forward's five kernels (amax + quantize of X, amax + quantize of W, GEMM) as one CUDA graph, "
                "replayed; L2 flushed before each replay",
        "value": round(statistics.mean(times) * 1e3, 2), "best": round(min(times) * 1e3, 2),
        "unit": "us per forward", "replays": iters}
    del graph, flush, x, w

    # ---- MoE expert forward: 8 experts x 1024 tokens, K 4096, N 1536 (up projection)
    E, T, K, N = 8, 8192, 4096, 1536
    x = I.normal_with_outliers(T, K, seed=1).to(dev)
    w = torch.stack([I.normal(N, K, seed=1000 + e, std=0.02) for e in range(E)]).to(dev)
    offs = [e * (T // E) for e in range(E + 1)]
    fl2 = 2.0 * T * N * K

    def c2(L):
        xc, xs, xsd, _ = L("quantize_1d", T * K, F.quantize_1d, x)
        wc, ws, wsd, _ = L("quantize_2d", E * N * K, F.quantize_2d, w)
        L("gemm_nvfp4_grouped", fl2, F.gemm_nvfp4, xc, xs, xsd, wc, ws, F.SCALE_2D, wsd, torch.bfloat16, E, offs)

    finish("moe_expert_fwd_8x1024x1536x4096", timed_calls(torch, dev, c2, iters),
           "X 8192x4096 N(0,1)+0.1% x50 (tokens in expert order, 1024 per expert), W_up 8x1536x4096 "
           "N(0,0.02); quantize X (1D) and W (2D, per expert), grouped NVFP4 GEMM bf16 out",
           lambda k: round(fl2 / (per_iter_ms(k) * 1e-3) / 1e12, 1), "TFLOP/s (GEMM FLOPs / forward time)")
    del x, w

    # ---- backward requantization: dY 8192 x 4096, X 8192 x 4096, W 4096 x 4096
    M, K, N = 8192, 4096, 4096
    seed, signs = I.sr_seed(2), I.rht_signs(2)
    dy = I.student_t(M, N, seed=2).to(dev)
    xc, xs, xsd, _ = F.quantize_1d(I.normal(M, K, seed=22).to(dev))
    wc, ws, wsd, _ = F.quantize_2d(I.normal(N, K, seed=23, std=0.02).to(dev))
    fl3 = 2.0 * M * N * K

    def c3(L):
        g, gt = L("requant_bf16_dual", M * N, F.requant_bf16_dual, dy, 1, signs, F.SR, seed, F.TAG_DY_ROWS,
                  F.TAG_DY_T)
        wt = L("requant_nvfp4_2d", N * K, F.requant_mxfp8, F.IN_NVFP4_2D, wc, ws, wsd, N, K, 1, 0, 0, F.SR, seed,
               F.TAG_WT)
        xt = L("requant_nvfp4_1d", M * K, F.requant_mxfp8, F.IN_NVFP4_1D, xc, xs, xsd, M, K, 1, 1, signs, F.SR,
               seed, F.TAG_XT)
        L("gemm_mxfp8_dgrad", fl3, F.gemm_mxfp8, g[0], g[1], wt[0], wt[1], torch.bfloat16)
        L("gemm_mxfp8_wgrad", fl3, F.gemm_mxfp8, gt[0], gt[1], xt[0], xt[1], torch.float32)

    finish("backward_requant_8192x4096x4096", timed_calls(torch, dev, c3, iters),
           "dY 8192x4096 Student-t(3)*1e-3, X 8192x4096 N(0,1) (NVFP4 1D), W 4096x4096 N(0,0.02) (NVFP4 2D); "
           "requants to MXFP8 with SR (dY rowwise + transposed with RHT16 from one read, X_q^T with RHT16, "
           "W_q^T), dgrad bf16 + wgrad fp32",
           lambda k: round(2 * fl3 / (per_iter_ms(k) * 1e-3) / 1e12, 1),
           "TFLOP/s (dgrad + wgrad FLOPs / backward time incl. requants)")
    del dy, xc, xs, wc, ws

    # ---- 2D weight quantize + GEMM sweep: W 14336 x 4096, X M x 4096, M in {1024, 4096, 16384}
    N, K = 14336, 4096
    w = I.normal(N, K, seed=33, std=0.02).to(dev)
    xs_ = {m: I.normal(m, K, seed=3).to(dev) for m in (1024, 4096, 16384)}
    wq = F.quantize_2d(w)

    def c4(L):
        L("quantize_2d", N * K, F.quantize_2d, w)
        for m, xm in xs_.items():
            xc, xs, xsd, _ = L(f"quantize_1d_M{m}", m * K, F.quantize_1d, xm)
            L(f"gemm_nvfp4_M{m}", 2.0 * m * N * K, F.gemm_nvfp4, xc, xs, xsd, wq[0], wq[1], F.SCALE_2D, wq[2],
              torch.bfloat16)

    finish("wq2d_gemm_sweep_14336x4096", timed_calls(torch, dev, c4, iters),
           "W 14336x4096 N(0,0.02) (2D quantize), X Mx4096 N(0,1) for M in 1024/4096/16384 (1D quantize), "
           "NVFP4 GEMM bf16 out",
           lambda k: round(2.0 * 16384 * N * K / (k["gemm_nvfp4_M16384"][1] / iters * 1e-3) / 1e12, 1),
           "TFLOP/s (NVFP4 GEMM at M=16384)", traffic_kinds=("gemm_nvfp4_M16384",))
    return out


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
    # and the host wall clock bracket the loop, which runs as many steps as the device-timed region
    # (the first step's input copy and the last step's result copy have nothing to overlap with).
    e2e_steps = max(1, args.steps)
    copy = torch.cuda.Stream(device=dev)          # host -> device
    copy_out = torch.cuda.Stream(device=dev)      # device -> host
    comp = torch.cuda.current_stream(dev)
    dbuf = [[torch.empty_like(t, device=dev) for t in host] for _ in range(2)]
    outs_host = None
    h2d = sum(t.numel() * t.element_size() for t in host)
    d2h = 0

    def e2e_loop(nsteps):
        # Each input has its own ready event and each call waits only for the inputs it reads
        # (StreamTap), and each result is copied out once the call that makes it is done, so
        # the first step starts after its first input's copy and the last step's earlier
        # results leave while it runs.
        nonlocal outs_host, d2h
        in_ready = [[torch.cuda.Event() for _ in host] for _ in range(2)]
        buf_free = [torch.cuda.Event() for _ in range(2)]
        out_done = torch.cuda.Event()

        def load(b):
            with torch.cuda.stream(copy):
                for d, hsrc, ev in zip(dbuf[b], host, in_ready[b]):
                    d.copy_(hsrc, non_blocking=True)
                    ev.record(copy)

        load(0)
        for i in range(nsteps):
            b = i % 2
            tap = StreamTap(torch.cuda.Event, comp, dbuf[b], in_ready[b])
            outs = mlp_step(F, torch, dbuf[b], tap, seed, signs)
            tap.finish()
            buf_free[b].record(comp)
            out_done.record(comp)
            if i + 1 < nsteps:
                nb = (i + 1) % 2
                if i >= 1:
                    copy.wait_event(buf_free[nb])
                load(nb)
            with torch.cuda.stream(copy_out):
                if outs_host is None:
                    outs_host = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
                for oh, o in zip(outs_host, outs):
                    copy_out.wait_event(tap.ready(o) or out_done)
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
    region_s = ms * 1e-3
    kernels = summarize_kernels(kinds, peaks, peak_src, region_s)
    dom = max(kinds.items(), key=lambda kv: kv[1][1])[0]
    roof = roofline_of(kernels, dom)
    value = STEP_FLOPS / (per_step * 1e-3) / 1e12
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4(e2m1,e4m3 scale)/mxfp8(e4m3,e8m0) x fp32-accum",
        "data": "synthetic (seeded bf16: X N(0,1)+0.1% x50 outliers, W N(0,0.02), dY Student-t(3)*1e-3)",
        "config": step_config(world),
        "roofline": roof,
        "kernels": kernels,
        "e2e": {"value": round(STEP_FLOPS / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": round(e2e_ms, 3), "event_ms": round(e2e_event_ms, 3),
                "wall_ms": round(e2e_wall_ms, 3)},
        "gpu_launches": int(sum(LAUNCHES_PER_STEP.values()) * args.steps),
        "clocks": clocks,
        "timed_region_s": round(region_s, 4),
        "per_token_4over6": {
            "what": "the same step with the activations quantized per token row with 4/6 block scales "
                    "(one pass, no activation amax), per-row outer scales through both GEMM epilogues "
                    "and the X^T requantizations",
            "value": round(STEP_FLOPS / (r_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "ms_per_step": round(r_ms, 4), "steps": r_steps, "warmup": 3,
            "gpu_launches": int(sum(LAUNCHES_PER_STEP_ROWS.values()) * r_steps),
            # traffic: only the kernels this form shares with the per-tensor step
            "kernels": summarize_kernels(rlog.totals(), peaks, peak_src, r_ms * r_steps * 1e-3,
                                         ("gemm_mxfp8", "quantize_2d", "requant_nvfp4_2d")),
        },
    }
    with ClockSampler(smi_id) as clk2:
        res["configs"] = configs_section(F, torch, dev, peaks, peak_src)
        res["combine_codec"] = combine_section(F, torch, dev, peaks)
        res["mxfp4_vs_nvfp4"] = format_section(F, torch, dev, peaks)
    res["clocks_other_sections"] = clk2.summary()
    res["targets"] = targets(res)
    if world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(args.cpu_sample)
        for name, rec in res["configs"].items():
            rec["cpu_baseline"] = cpu_baseline_config(name, rec)
    if dist is not None:
        dist.destroy_process_group()
    return res


def step_config(world):
    return {"workload": WORKLOAD, "tokens": M_TOK, "d_model": D_MODEL, "ffn": F_FFN,
            "step": "MLP block fwd (2 NVFP4 GEMMs) + bwd (4 MXFP8 GEMMs, SR, RHT16 on wgrad)",
            "l2": "no flush: per-step working set > 4 GB >> 129 MB L2", "parallelism": f"replicas x{world}"}


def targets(res):
    """The stated targets against the measured figures: the NVFP4 GEMM at the largest shape
    (X 16384 x 4096 times W 14336 x 4096) at >= 60% of the dense FP4 peak, and each quantize /
    requantize kernel at >= 70% of HBM bandwidth (of the measured copy rate)."""
    sweep = res["configs"]["wq2d_gemm_sweep_14336x4096"]["kernels"]
    g = sweep["gemm_nvfp4_M16384"]
    hbm = {}
    for where, kern in (("step", res["kernels"]), ("sweep", sweep),
                        ("backward_requant", res["configs"]["backward_requant_8192x4096x4096"]["kernels"])):
        for kind, k in kern.items():
            if not kind.startswith("gemm"):
                hbm[f"{where}:{kind}"] = k["frac"]
    return {"nvfp4_gemm_largest": {"kernel": "gemm_nvfp4_M16384 (16384x14336x4096, bf16 out)",
                                   "achieved": g["achieved"], "unit": g["unit"], "peak": g["peak"],
                                   "peak_source": g["peak_source"], "frac": g["frac"], "target": 0.60,
                                   "met": g["frac"] >= 0.60},
            "hbm_kernels": {"target": 0.70, "frac": hbm,
                            "met": sorted(k for k, v in hbm.items() if v >= 0.70),
                            "missed": sorted(k for k, v in hbm.items() if v < 0.70)}}


# ---------------------------------------------------------------------------- CPU oracle
def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def _timed(fn):
    t = time.perf_counter()
    out = fn()
    return out, time.perf_counter() - t


def _gemm_time(deq_a, rows_a_full, deq_b, rows_b_full, k_scale=1.0):
    """Dequantize a row sample of each operand and multiply (float64); extrapolate linearly to
    the full operands (dequant per row, product per row pair, both per unit of K)."""
    A, ta = _timed(deq_a)
    B, tb = _timed(deq_b)
    _, tm = _timed(lambda: A @ B.T)
    return (ta * rows_a_full / A.shape[0] + tb * rows_b_full / B.shape[0] +
            tm * (rows_a_full / A.shape[0]) * (rows_b_full / B.shape[0])) * k_scale


def _oracle_step(r):
    """The MLP step on a bounded sample: r rows of every operand, extrapolated to the full step."""
    import numpy as np
    import oracle as O
    from mxfp8_precision_numerics_gb300 import inputs as I

    M, D, Fh = M_TOK, D_MODEL, F_FFN
    r = max(16, int(r))
    seed, signs = I.sr_seed(SEED), I.rht_signs(SEED)
    xs = I.bf16_bits(I.normal_with_outliers(r, D, seed=SEED))
    w1s = I.bf16_bits(I.normal(r, D, seed=41, std=0.02))
    w2s = I.bf16_bits(I.normal(r, Fh, seed=42, std=0.02))
    hs = I.bf16_bits(I.normal(r, Fh, seed=43))
    dys = I.bf16_bits(I.student_t(r, D, seed=44))
    dhs = I.bf16_bits(I.student_t(r, Fh, seed=45))
    est = 0.0
    (xc, xsc, _, xsd), t = _timed(lambda: O.quantize_1d(xs)); est += t * M / r
    (w1c, w1t, _, w1d), t = _timed(lambda: O.quantize_2d(w1s)); est += t * Fh / r
    (ac, asc, _, ad), t = _timed(lambda: O.quantize_1d(hs)); est += t * M / r
    (w2c, w2t, _, w2d), t = _timed(lambda: O.quantize_2d(w2s)); est += t * D / r
    est += _gemm_time(lambda: O.dequant_nvfp4(xc, xsc, 1, xsd), M, lambda: O.dequant_nvfp4(w1c, w1t, 2, w1d), Fh)
    est += _gemm_time(lambda: O.dequant_nvfp4(ac, asc, 1, ad), M, lambda: O.dequant_nvfp4(w2c, w2t, 2, w2d), D)
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
        _, t = _timed(lambda: O.requant_mxfp8(kind, data, sc, sd, rows, cols, tr, rht, signs, O.SR, seed, 1,
                                              out_rows=(0, n_out)))
        est += t * (f_or * f_oc) / (n_out * (rows if tr else cols))
    # MXFP8 GEMMs: dequant + product of sampled rows (random E4M3 bytes: the work does not
    # depend on the values), extrapolated
    e4 = np.random.default_rng(0).integers(0, 0x7E, (r, Fh), dtype=np.uint8)
    e8 = np.full((r, Fh // 32), 127, np.uint8)
    for rows_a, rows_b, k in ((M, Fh, D), (D, Fh, M), (M, D, Fh), (Fh, D, M)):
        kk = min(k, Fh)
        deq = lambda: O.dequant_mxfp8(e4[:, :kk], e8[:, :kk // 32])
        est += _gemm_time(deq, rows_a, deq, rows_b, k / kk)
    return {"total": est}


def _oracle_config(name, r):
    """One of the four other workloads on a bounded sample (r rows), extrapolated."""
    import numpy as np
    import oracle as O
    from mxfp8_precision_numerics_gb300 import inputs as I
    r = max(16, int(r) // 16 * 16)
    if name == "linear_fwd_256x512":
        xb = I.bf16_bits(I.normal_with_outliers(256, 512, seed=0))
        wb = I.bf16_bits(I.normal(256, 512, seed=100, std=0.02))
        n, t0 = 0, time.perf_counter()
        while n < 3 or time.perf_counter() - t0 < 0.5:
            xc, xs, _, xsd = O.quantize_1d(xb)
            wc, ws, _, wsd = O.quantize_2d(wb)
            O.gemm_nvfp4(xc, xs, 1, xsd, wc, ws, 2, wsd)
            n += 1
        return {"total": (time.perf_counter() - t0) / n}
    if name == "moe_expert_fwd_8x1024x1536x4096":
        E, T, K, N = 8, 8192, 4096, 1536
        xb = I.bf16_bits(I.normal_with_outliers(r, K, seed=1))
        wb = I.bf16_bits(I.normal(N, K, seed=1000, std=0.02))
        (xc, xs, _, xsd), tq = _timed(lambda: O.quantize_1d(xb))
        (wc, ws, _, wsd), tw = _timed(lambda: O.quantize_2d(wb[:r]))
        wq = O.quantize_2d(wb)
        tg = _gemm_time(lambda: O.dequant_nvfp4(xc, xs, 1, xsd), T // E,
                        lambda: O.dequant_nvfp4(wq[0], wq[1], 2, wq[3]), N) * E
        return {"total": tq * T / r + tw * E * N / r + tg}
    if name == "backward_requant_8192x4096x4096":
        M, K, N = 8192, 4096, 4096
        seed, signs = I.sr_seed(2), I.rht_signs(2)
        est = 0.0
        dyr = I.bf16_bits(I.student_t(r, N, seed=2))
        dyc = I.bf16_bits(I.student_t(M, 32, seed=3))      # 32 columns: 32 output rows of dY^T
        xq = O.quantize_1d(I.bf16_bits(I.normal(M, 32, seed=22)))
        wq = O.quantize_2d(I.bf16_bits(I.normal(N, 32, seed=23, std=0.02)))
        _, t = _timed(lambda: O.requant_mxfp8(O.IN_BF16, dyr, None, 1.0, r, N, False, False, 0, O.SR, seed, 2))
        est += t * M / r
        _, t = _timed(lambda: O.requant_mxfp8(O.IN_BF16, dyc, None, 1.0, M, 32, True, True, signs, O.SR, seed, 3))
        est += t * N / 32
        _, t = _timed(lambda: O.requant_mxfp8(O.IN_NVFP4_1D, xq[0], xq[1], xq[3], M, 32, True, True, signs, O.SR,
                                              seed, 4))
        est += t * K / 32
        _, t = _timed(lambda: O.requant_mxfp8(O.IN_NVFP4_2D, wq[0], wq[1], wq[3], N, 32, True, False, 0, O.SR,
                                              seed, 1))
        est += t * K / 32
        rng = np.random.default_rng(0)
        e4a = rng.integers(0, 0x7E, (r, M), dtype=np.uint8)
        e4b = rng.integers(0, 0x7E, (1024, M), dtype=np.uint8)
        e8a = np.full((r, M // 32), 127, np.uint8)
        e8b = np.full((1024, M // 32), 127, np.uint8)
        # dgrad (K = 4096) and wgrad (K = 8192), random E4M3 bytes
        est += _gemm_time(lambda: O.dequant_mxfp8(e4a[:, :N], e8a[:, :N // 32]), M,
                          lambda: O.dequant_mxfp8(e4b[:, :N], e8b[:, :N // 32]), K)
        est += _gemm_time(lambda: O.dequant_mxfp8(e4a, e8a), N, lambda: O.dequant_mxfp8(e4b, e8b), K)
        return {"total": est}
    if name == "wq2d_gemm_sweep_14336x4096":
        N, K = 14336, 4096
        wb = I.bf16_bits(I.normal(1024, K, seed=33, std=0.02))
        (wc, ws, _, wsd), tw = _timed(lambda: O.quantize_2d(wb[:r]))
        wq = O.quantize_2d(wb)
        out = {"quantize_2d": tw * N / r}
        xb = I.bf16_bits(I.normal(r, K, seed=3))
        (xc, xs, _, xsd), tq = _timed(lambda: O.quantize_1d(xb))
        for m in (1024, 4096, 16384):
            out[f"gemm_M{m}"] = _gemm_time(lambda: O.dequant_nvfp4(xc, xs, 1, xsd), m,
                                           lambda: O.dequant_nvfp4(wq[0], wq[1], 2, wq[3]), N)
            out[f"quantize_1d_M{m}"] = tq * m / r
        out["total"] = sum(out.values())
        return out
    raise ValueError(name)


def _oracle_worker(name, rows):
    return _oracle_step(rows) if name == "step" else _oracle_config(name, rows)


def _spawn_oracle(name, rows, repeat, procs):
    """`procs` single-threaded oracle processes at once (fresh interpreters: nothing forked after
    CUDA), each timing `repeat` samples; returns their estimates and the wall time."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-worker", name, "--oracle-rows", str(rows),
           "--oracle-repeat", str(repeat)]
    t = time.perf_counter()
    ps = [subprocess.Popen(cmd, env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
          for _ in range(procs)]
    outs = []
    for p in ps:
        try:
            so, se = p.communicate(timeout=1800)
        except subprocess.TimeoutExpired:
            p.kill()
            raise RuntimeError("oracle worker timed out")
        if p.returncode != 0:
            tail = se.strip().splitlines()[-1] if se.strip() else "no output"
            raise RuntimeError("oracle worker failed: " + tail)
        outs.append(json.loads(so.strip().splitlines()[-1]))
    return outs, time.perf_counter() - t


def _cpu_estimates(name, rows):
    """Estimated full-workload seconds (dict of parts) on one core and on all cores. All cores:
    one single-threaded process per core, each on its own sample at the same time; the workload
    splits by rows, so its time is the median per-process estimate over the process count."""
    ncores = os.cpu_count() or 1
    one, wall1 = _spawn_oracle(name, rows, 1, 1)
    many, walln = _spawn_oracle(name, rows, 1, ncores)
    est1 = one[0][0]
    keys = est1.keys()
    estn = {k: statistics.median(o[0][k] for o in many) / ncores for k in keys}
    return est1, estn, ncores, wall1 + walln


def cpu_baseline(sample_rows):
    """The oracle on a bounded sample of the step, on one core and on all cores."""
    try:
        est1, estn, ncores, wall = _cpu_estimates("step", sample_rows)
    except (RuntimeError, subprocess.TimeoutExpired) as e:
        return {"value": None, "unit": "TFLOP/s", "cores": 0, "kind": "oracle", "sample": str(e)}
    return {"value": round(STEP_FLOPS / estn["total"] / 1e12, 6), "unit": "TFLOP/s", "cores": ncores,
            "kind": "oracle", "cpu_model": cpu_model(),
            "sample": (f"{sample_rows} rows of every operand of one step (quantize; requant of 16 output rows; "
                       f"GEMM dequant + float64 product of sampled rows; random E4M3 bytes for the MXFP8 "
                       f"GEMM operands), extrapolated linearly to the full step; all cores: one single-threaded "
                       f"process per core on its own sample at once; {wall:.1f} s wall in all"),
            "est_step_s": round(estn["total"], 2),
            "one_core": {"value": round(STEP_FLOPS / est1["total"] / 1e12, 6), "unit": "TFLOP/s", "cores": 1,
                         "est_step_s": round(est1["total"], 2)}}


CONFIG_SAMPLE_ROWS = {"linear_fwd_256x512": 256, "moe_expert_fwd_8x1024x1536x4096": 64,
                      "backward_requant_8192x4096x4096": 32, "wq2d_gemm_sweep_14336x4096": 64}


def cpu_baseline_config(name, rec):
    """The oracle on a bounded sample of one of the other workloads, in that workload's unit."""
    rows = CONFIG_SAMPLE_ROWS[name]
    try:
        est1, estn, ncores, wall = _cpu_estimates(name, rows)
    except (RuntimeError, subprocess.TimeoutExpired) as e:
        return {"value": None, "unit": rec["unit"], "cores": 0, "kind": "oracle", "sample": str(e)}

    def val(est):
        if name == "linear_fwd_256x512":
            return round(est["total"] * 1e6, 1)
        if name == "moe_expert_fwd_8x1024x1536x4096":
            return round(2.0 * 8192 * 1536 * 4096 / est["total"] / 1e12, 6)
        if name == "backward_requant_8192x4096x4096":
            return round(2 * 2.0 * 8192 * 4096 * 4096 / est["total"] / 1e12, 6)
        return round(2.0 * 16384 * 14336 * 4096 / est["gemm_M16384"] / 1e12, 6)

    sample = ("the whole forward, repeated" if name == "linear_fwd_256x512" else
              f"{rows} rows of each operand (transposed requants: 32 input columns; GEMMs: dequant + "
              f"float64 product of a row sample, random E4M3 bytes for MXFP8 operands), extrapolated linearly")
    return {"value": val(estn), "unit": rec["unit"], "cores": ncores, "kind": "oracle", "cpu_model": cpu_model(),
            "sample": sample + f"; all cores: one single-threaded process per core at once; {wall:.1f} s wall",
            "one_core": {"value": val(est1), "cores": 1}}


def run_reference(args, rank):
    """The reference arm: the CPU oracle on a bounded sample of the same step, per step, one
    single-threaded process per host core (the step splits by rows)."""
    if rank != 0:
        return None
    rows = max(16, args.cpu_sample // 4)
    ncores = os.cpu_count() or 1
    outs, wall = _spawn_oracle("step", rows, args.warmup + args.steps, ncores)
    per_step = [statistics.median(o[i]["total"] for o in outs) / ncores for i in range(args.warmup + args.steps)]
    est = statistics.median(per_step[args.warmup:])
    value = STEP_FLOPS / est / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(est * 1e3, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64/f32 (CPU oracle)",
        "data": "synthetic (same seeded generators)",
        "config": step_config(1),
        "cpu_baseline": {"kind": "oracle", "cores": ncores, "value": round(value, 6), "cpu_model": cpu_model(),
                         "sample": (f"{rows} sampled rows per operand per step on each of {ncores} single-threaded "
                                    f"processes at once, extrapolated to the full step; "
                                    f"{args.warmup + args.steps} samples per process in {wall:.1f} s")},
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
    ap.add_argument("--oracle-worker", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--oracle-rows", type=int, default=512, help=argparse.SUPPRESS)
    ap.add_argument("--oracle-repeat", type=int, default=1, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_worker is not None:
        print(json.dumps([_oracle_worker(args.oracle_worker, args.oracle_rows) for _ in range(args.oracle_repeat)]))
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
