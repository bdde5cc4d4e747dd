"""The benchmark's host arithmetic on the CPU: which tensor peak a GEMM rate is divided by, the
achieved rate and roofline fraction of each call kind, the DRAM-traffic lookup (only for kinds
timed at the captured shapes, and only while the kernel sources are the captured ones), the
stated targets and the shape of the step's config record."""
import hashlib
import json
import os

import pytest

import bench

PEAKS = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1500.0}


def test_gemm_peak_burst_or_sustained_by_region():
    p, how = bench.gemm_peak(PEAKS, fp4=True, region_s=0.1)
    assert p == 2000.0 * bench.RATIO_FP4 and how == "bf16 burst x 6"
    p, how = bench.gemm_peak(PEAKS, fp4=False, region_s=5.0)
    assert p == 1500.0 * bench.RATIO_FP8 and how == "bf16 sustained x 2"
    # the boundary: 2 s and longer is a sustained region
    assert bench.gemm_peak(PEAKS, fp4=False, region_s=2.0)[0] == 1500.0 * 2


def test_summarize_kernels_rates_and_fractions():
    # (launches, total ms, units): GEMM units are FLOPs, the others elements
    kinds = {"gemm_nvfp4": (2, 1.0, 4.0e12), "quantize_1d": (4, 2.0, 1.0e9), "requant_bf16_dual": (1, 0.5, 2.0e8)}
    k = bench.summarize_kernels(kinds, PEAKS, "measured", region_s=0.5, traffic_kinds=())
    g = k["gemm_nvfp4"]
    assert g["avg_ms"] == 0.5 and g["achieved"] == pytest.approx(4000.0)
    assert g["peak"] == pytest.approx(12000.0) and g["frac"] == pytest.approx(4000.0 / 12000.0, abs=1e-4)
    assert g["peak_source"] == "measured bf16 burst x 6"
    q = k["quantize_1d"]
    gbs = 1.0e9 * bench.BYTES_PER_ELEM["quantize_1d"] / 2.0e-3 / 1e9
    assert q["achieved"] == pytest.approx(gbs, rel=1e-4) and q["frac"] == pytest.approx(gbs / 6000.0, rel=1e-3)
    assert q["unit"] == "GB/s (amax + quantize passes)"
    d = k["requant_bf16_dual"]
    # rowwise and transposed outputs from one read of bf16: 2 + 2 (1 + 1/32) bytes per element
    assert bench.BYTES_PER_ELEM["requant_bf16_dual"] == pytest.approx(2.0 + 2.0 * (1 + 1 / 32))
    assert d["unit"] == "GB/s"
    assert all(v["traffic"] is None for v in k.values())


def test_sweep_kinds_use_their_base_bytes():
    k = bench.summarize_kernels({"quantize_1d_M4096": (1, 1.0, 1.0e9)}, PEAKS, traffic_kinds=())
    assert k["quantize_1d_M4096"]["achieved"] == pytest.approx(1.0e9 * bench.BYTES_PER_ELEM["quantize_1d"] / 1e-3 / 1e9,
                                                               rel=1e-4)


def test_traffic_only_for_listed_kinds(monkeypatch):
    monkeypatch.setattr(bench, "ncu_traffic", lambda kind: 123)
    kinds = {"gemm_mxfp8": (1, 1.0, 1e12), "quantize_2d": (1, 1.0, 1e6)}
    k = bench.summarize_kernels(kinds, PEAKS, traffic_kinds=("gemm_mxfp8",))
    assert k["gemm_mxfp8"]["traffic"] == 123 and k["quantize_2d"]["traffic"] is None
    k = bench.summarize_kernels(kinds, PEAKS)            # None: the step itself, every kind
    assert k["gemm_mxfp8"]["traffic"] == 123 and k["quantize_2d"]["traffic"] == 123


def test_ncu_traffic_follows_the_sources(tmp_path, monkeypatch):
    csrc = tmp_path / "mxfp8_precision_numerics_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "k.cu").write_bytes(b"kernel v1")
    sha = hashlib.sha256(b"kernel v1").hexdigest()[:16]
    rec = {"k": {"sources": ["k.cu"], "source_sha": sha, "captures": ["c"], "dram_bytes_per_launch": 777}}
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.ncu_traffic("k") == 777
    assert bench.ncu_traffic("other") is None
    (csrc / "k.cu").write_bytes(b"kernel v2")             # the kernel changed since the capture
    assert bench.ncu_traffic("k") is None


def test_committed_traffic_table_names_its_captures():
    path = os.path.join(bench.ROOT, "profiles", "ncu_traffic.json")
    with open(path) as f:
        rec = json.load(f)
    assert "-c 1" in rec["_about"] and "--clock-control none" in rec["_about"]
    for kind, v in rec.items():
        if kind.startswith("_"):
            continue
        assert v["captures"] and v["dram_bytes_per_launch"] > 0 and len(v["source_sha"]) == 16


def test_roofline_of_and_targets():
    kern = bench.summarize_kernels({"gemm_nvfp4_M16384": (1, 1.0, 7.2e12), "quantize_2d": (1, 1.0, 1e9),
                                    "gemm_nvfp4_M1024": (1, 1.0, 1e11)}, PEAKS, traffic_kinds=())
    r = bench.roofline_of(kern, "gemm_nvfp4_M16384")
    assert r["bound"] == "tensor" and r["frac"] == kern["gemm_nvfp4_M16384"]["frac"]
    assert bench.roofline_of(kern, "quantize_2d")["bound"] == "hbm"
    res = {"kernels": {"quantize_1d": {"frac": 0.72}, "requant_nvfp4_1d": {"frac": 0.24}, "gemm_mxfp8": {"frac": 0.7}},
           "configs": {"wq2d_gemm_sweep_14336x4096": {"kernels": kern},
                       "backward_requant_8192x4096x4096": {"kernels": {"requant_bf16_dual": {"frac": 0.35}}}}}
    t = bench.targets(res)
    g = t["nvfp4_gemm_largest"]
    assert g["frac"] == kern["gemm_nvfp4_M16384"]["frac"] and g["met"] == (g["frac"] >= 0.60)
    h = t["hbm_kernels"]
    assert "step:quantize_1d" in h["met"] and "step:requant_nvfp4_1d" in h["missed"]
    assert "backward_requant:requant_bf16_dual" in h["missed"]
    assert not any(k.endswith("gemm_mxfp8") or "gemm_nvfp4" in k for k in h["frac"])


def test_step_config_names_the_workload():
    c = bench.step_config(4)
    assert c["workload"] == bench.WORKLOAD and c["parallelism"] == "replicas x4"
    assert (c["tokens"], c["d_model"], c["ffn"]) == (16384, 4096, 16384)
    # six GEMMs of 2 M D F FLOPs each per step
    assert bench.STEP_FLOPS == 6 * 2.0 * 16384 * 4096 * 16384


def test_stream_tap_waits_per_input_and_marks_outputs():
    import torch

    class Ev:
        def __init__(self, name=""):
            self.name, self.on = name, None

        def record(self, stream):
            self.on = stream

    class Stream:
        def __init__(self):
            self.waits = []

        def wait_event(self, ev):
            self.waits.append(ev.name)

    comp = Stream()
    buf = torch.zeros(64, dtype=torch.bfloat16)
    x, w1, w2, dy = buf[:16], buf[16:32], buf[32:48], buf[48:]
    ready = [Ev(n) for n in ("x", "w1", "w2", "dy")]
    made = []

    def new_event():
        made.append(Ev("call%d" % len(made)))
        return made[-1]

    tap = bench.StreamTap(new_event, comp, [x, w1, w2, dy], ready)
    y = torch.zeros(4)
    # a call on a view of x waits for x alone; a second use waits for nothing more
    out = tap.wrap("k", 1, lambda t, s: (y, s), x[2:5], 3)
    assert comp.waits == ["x"] and out[0] is y and tap.ready(y) is made[0] and made[0].on is comp
    tap.wrap("k", 1, lambda t: None, x)
    assert comp.waits == ["x"]
    # nested arguments and keywords count; w1 and dy overlap, w2 does not
    tap.wrap("k", 1, lambda *a, **k: None, [w1[:1], (3,)], amax_in=dy[-1:])
    assert comp.waits == ["x", "w1", "dy"]
    assert tap.ready(torch.zeros(1)) is None
    tap.finish()
    assert comp.waits == ["x", "w1", "dy", "w2"]
