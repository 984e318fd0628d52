"""bench.py's reference arm on the host: one JSON line with the contract's keys
(the oracle timed on the host cores, on a bounded sample of the workload)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--config", "tiny", "--steps", "2", "--warmup", "0"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["higher_is_better"] is True and d["n_gpus"] == 1 and d["warmup"] >= 3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith("tiny")
    # ms_per_step is the measured sample step, so steps x ms_per_step is the timed region
    assert abs(d["ms_per_step"] - 1e3 * d["cpu_baseline"]["sample_s"]) < 1e-6
    assert d["timing"]["estimated_full_step_ms"] > 0


def test_layout_metrics_eta_matches_the_oracle():
    """bench.py's eta (mean over max of the count matrix's column sums) is the
    oracle's imbalance_eta, and its padding fraction follows the tile rule."""
    import importlib.util
    import numpy as np
    sys.path.insert(0, ROOT)
    import oracle
    import synth
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    rng = np.random.default_rng(3)
    for n_ep in (2, 8, 64):
        C = rng.integers(0, 50, size=(n_ep, n_ep))
        C[0, 0] += 1
        cfg = synth.CONFIGS["tiny"].with_(n_ep=n_ep, E=64)
        counts = rng.integers(0, 300, size=64)
        got = b.layout_metrics(cfg, counts, C)
        assert got["eta"] == oracle.imbalance_eta(C)
    # tiles: 300 rows -> 128 + 128 + a 64-row half tile; 200 -> 128 + 128; 0 -> nothing
    assert b.tile_rows([300, 200, 0, 64, 65]) == 320 + 256 + 0 + 64 + 128


def test_tensor_peak_rule():
    """The sustained bf16 peak (seconds of back-to-back GEMMs at the power limit)
    is the denominator only for a timed region that long which also ran capped
    below the top clock; otherwise the burst peak."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    pk = {"bf16_tflops": 1749.0, "bf16_tflops_sustained": 1350.5, "source": "measured"}
    capped_low = {"power_cap_share": 0.9, "sm_mhz": 1500.0, "sm_max_mhz": 2032.0}
    capped_top = {"power_cap_share": 0.9, "sm_mhz": 2032.0, "sm_max_mhz": 2032.0}
    assert b._tensor_peak(pk, capped_low, 2.5)[0] == 1350.5
    assert b._tensor_peak(pk, capped_low, 0.05)[0] == 1749.0   # a short region: burst
    assert b._tensor_peak(pk, capped_top, 2.5)[0] == 1749.0    # capped but at the top clock
    assert b._tensor_peak(pk, {"power_cap_share": 0.2, "sm_mhz": 1500.0,
                               "sm_max_mhz": 2032.0}, 2.5)[0] == 1749.0
    assert b._tensor_peak(pk, None, 5.0)[0] == 1749.0


def test_cpu_baseline_runs_bounded_samples():
    """bench.py's cpu_baseline leg on the host: the oracle's sample repeated
    until the requested seconds of host work (bounded by a run count), its
    median reported with the runs and seconds it took."""
    import importlib.util
    import torch
    sys.path.insert(0, ROOT)
    import synth
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    cfg = synth.CONFIGS["tiny"].with_(T=256)
    x = synth.make_x(cfg)
    W_r, lbias = synth.make_router(cfg)
    W1, W3, W2 = synth.make_expert_weights(cfg)

    import types
    # the layer's packed weights: W13 rows interleaved in 128-row blocks
    W13 = torch.stack([torch.cat([torch.cat([W1[e, i:i + 128], W3[e, i:i + 128]])
                                  for i in range(0, cfg.f, 128)]) for e in range(cfg.E)])
    packed = types.SimpleNamespace(W13=W13, W2=W2)
    got = b.cpu_baseline(cfg, x, W_r, lbias, packed, reps=2, min_s=0.2, max_reps=6)
    assert 2 <= got["sample_runs"] <= 6 and got["host_s"] > 0
    assert got["kind"] == "oracle" and got["value"] > 0 and got["unit"] == "tokens/s"
    assert got["sample_runs"] == 6 or got["host_s"] >= 0.2


def test_serving_ridge_reasoning():
    """The pages' serving ridge ("Expert parallelism", "Serving"): an expert's
    product with n tokens does 2 n d d_e FLOPs per weight matrix and reads d d_e
    2-byte weights, about n FLOPs per byte; an H100 needs 989/3.35 ~ 295 FLOPs
    per byte, so about 300 tokens per expert, 300 E / k ~ 9,600 tokens for
    DeepSeek-V3.  The benchmark's FLOP and weight-byte models give the same
    intensity, and its roofline puts a layer on the tensor side exactly when the
    rows per expert pass the ridge of the peaks it divides by."""
    import importlib.util
    sys.path.insert(0, ROOT)
    import numpy as np
    import synth
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    assert round(989 / 3.35) == 295
    assert 300 * 256 // 8 == 9600
    for n in (4, 64, 288, 1024):
        cfg = synth.CONFIGS["dsv3"].with_(T=n * 256 // 8, has_shared=0)
        counts = np.full(cfg.E, n)
        flops = b._algorithmic(cfg, counts)["ffn_flops"]
        weight_bytes = cfg.E * 3 * cfg.d * cfg.f * 2
        assert flops / weight_bytes == n
        # the model's bytes also hold the activations, so its ridge sits a little above n
        ffn_bytes = b._ffn_bytes(cfg, counts)
        assert ffn_bytes > weight_bytes
        pk = {"hbm_gbs": 6503.1, "bf16_tflops": 1749.0, "bf16_tflops_sustained": 1350.5,
              "source": "measured"}
        line = b._roofline(cfg, 1.0, flops, ffn_bytes, pk, {}, 0.1)
        ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)   # ~269 FLOPs per byte
        assert line["bound"] == ("tensor" if flops / ffn_bytes >= ridge else "hbm")
        assert line["bound"] == ("tensor" if n >= 1024 else "hbm")   # 288 rows: at the ridge, HBM side
