"""Benchmark of the single-device MoE layer hot path on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

One step = one pass of the whole hot path over one batch of synthetic tokens:
router logits -> top-k route -> permute (expert-grouped buffer) -> simulated
expert-parallel layout (count matrix, offsets, packed send buffer) -> grouped
SwiGLU FFN (two tcgen05 grouped GEMMs) -> unpermute + gate + combine.

Prints ONE JSON line (rank 0).  Default workload: the Mixtral-8x7B-shaped layer
(T=4096, d=4096, E=8, f=14336, top-2, n_ep=8).  Inputs and weights are seeded
random draws resident in HBM before timing; L2 is flushed (a 512 MiB write, then a 256 MiB read)
between timed steps, outside the timed events.  With N > 1 (torchrun) every
rank runs an independent replica of the layer on its own batch (weak scaling,
no collective on the data path); the barrier and the max over ranks are for
timing only.

--impl reference times the oracle (fp64 numpy on the host cores) on a bounded
sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "MoE-layer tokens/s on 1 B300; grouped-FFN % BF16 peak; permute/combine % HBM"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


def _workload(cfg):
    s = (f"{cfg.name}: T={cfg.T} d={cfg.d} E={cfg.E} f={cfg.f} top-{cfg.k} {cfg.score_fn}"
         f" n_ep={cfg.n_ep}")
    if cfg.n_groups > 1:
        s += f" groups={cfg.n_groups}/top{cfg.topk_groups}"
    if cfg.has_shared:
        s += " +1 shared"
    if cfg.capacity:
        s += f" capacity={cfg.capacity}"
    return s


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _max_over_ranks(v, dev, world):
    """The largest of every rank's value (each rank's own when world == 1): the
    slowest replica sets the job's time."""
    if world <= 1:
        return float(v)
    t = torch.tensor([float(v)], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


class _Clocks:
    """SM clocks and throttle reasons during the timed region: NVML read every
    20 ms from a thread (the statistics), and nvidia-smi every 200 ms beside it
    (the raw record, kept as a file)."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # NVML clocks-event reason bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.thread = None
        self.samples = []
        # raw samples: MOE_BENCH_CLOCKS_DIR if set, else the temp directory
        base = os.environ.get("MOE_BENCH_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(base, f"moe_bench_clocks_rank{index}.csv")

    def _nvml_loop(self, stop):
        """Read-only NVML queries through the driver's libnvidia-ml (ctypes)."""
        import ctypes
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise RuntimeError("nvmlInit_v2 failed")
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) != 0:
                raise RuntimeError("nvmlDeviceGetHandleByIndex_v2 failed")
            reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            mhz, mx, bits = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
            if nv.nvmlDeviceGetMaxClockInfo(h, ctypes.c_int(1), ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            while not stop.is_set():
                if (nv.nvmlDeviceGetClockInfo(h, ctypes.c_int(1), ctypes.byref(mhz)) == 0 and
                        reasons_fn(h, ctypes.byref(bits)) == 0):
                    self.samples.append((float(mhz.value), int(bits.value)))
                stop.wait(0.02)
            nv.nvmlShutdown()
        except Exception as exc:  # no NVML: the nvidia-smi record alone
            self.nvml_error = f"{type(exc).__name__}: {exc}"
            return

    def start(self):
        import threading
        self._stop = threading.Event()
        self.thread = threading.Thread(target=self._nvml_loop, args=(self._stop,), daemon=True)
        self.thread.start()
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}",
                                          f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", "200"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def _smi_rows(self):
        if self.proc is None:
            return []
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        for ln in open(self.path):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[4:]))
            except ValueError:
                continue
        return rows

    def stop(self):
        if self.thread is not None:
            self._stop.set()
            self.thread.join(timeout=5)
        rows = self._smi_rows()
        if self.samples:
            mx = getattr(self, "max_mhz", max(m for m, _ in self.samples))
            reasons = sorted({n for _, b in self.samples for bit, n in self.REASONS.items()
                              if b & bit})
            cap = sum(1 for _, b in self.samples if b & 0x4) / len(self.samples)
            return {"sm_mhz": statistics.median(m for m, _ in self.samples), "sm_max_mhz": mx,
                    "reasons": reasons, "samples": len(self.samples),
                    "power_cap_share": cap, "smi_samples": len(rows),
                    "source": "NVML every 20 ms during the timed region (nvidia-smi every "
                              "200 ms beside it)"}
        if not rows:
            return None
        mx = max(r[1] for r in rows)
        extra = {"nvml_error": self.nvml_error} if getattr(self, "nvml_error", None) else {}
        load = [r for r in rows if r[0] > 0.3 * mx] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in load for i, v in enumerate(r[2][1:5])
                          if v.lower() == "active"})
        cap = sum(1 for r in load if r[2][4].lower() == "active") / len(load)
        return {"sm_mhz": statistics.median(r[0] for r in load), "sm_max_mhz": mx,
                "reasons": reasons, "samples": len(rows), "power_cap_share": cap,
                "source": "nvidia-smi every 200 ms during the timed region", **extra}


def _algorithmic(cfg, counts_np, gather=False):
    """Algorithmic FLOPs and bytes of one step (what the method must do).  With
    the gather path the permute moves no rows (GEMM 1 reads the token rows)."""
    kept = int(np.minimum(counts_np, cfg.capacity).sum()) if cfg.capacity else cfg.A
    rows_ffn = kept + (cfg.T if cfg.has_shared else 0)
    R = cfg.R
    b2 = 2  # bf16
    out = {
        "ffn_flops": 6.0 * cfg.d * cfg.f * rows_ffn,
        "router_bytes": cfg.T * cfg.d * b2 + cfg.d * cfg.E * 4 + cfg.T * cfg.E * 4,
        "route_bytes": cfg.T * cfg.E * 4 + cfg.A * 8,
        "permute_bytes": (0 if gather else cfg.T * cfg.d * b2 + R * cfg.d * b2)
                         + 4 * (2 * cfg.A + R + 2 * cfg.E),
        "layout_bytes": cfg.T * cfg.d * b2 + cfg.A * cfg.d * b2 + 4 * 4 * cfg.A,
        "combine_bytes": (kept + (cfg.T if cfg.has_shared else 0)) * cfg.d * b2
                         + cfg.T * cfg.d * b2 + 8 * cfg.A,
        "rows_ffn": rows_ffn,
    }
    return out


def tile_rows(kept, bm=128):
    """Rows the grouped GEMM computes for segments of `kept` rows: whole
    128-row tiles, except a last tile holding at most 64 rows, which runs as a
    64-row half tile."""
    kept = np.asarray(kept, np.int64)
    full, rem = kept // bm, kept % bm
    return int((full * bm + np.where(rem == 0, 0, np.where(rem <= bm // 2, bm // 2, bm))).sum())


def layout_metrics(cfg, counts, C):
    """The layer's load metrics: rows per expert, the drop and padding
    fractions, and eta = mean over max of the ranks' received rows (the column
    sums of the count matrix): the useful fraction of the group's expert
    compute ("Expert parallelism", "Load imbalance becomes idle time")."""
    counts = np.asarray(counts, np.int64)
    kept = np.minimum(counts, cfg.capacity) if cfg.capacity else counts
    loads = np.asarray(C, np.float64).sum(axis=0)
    rows_kept = int(kept.sum()) + (cfg.T if cfg.has_shared else 0)
    rows_tiled = tile_rows(kept) + (tile_rows([cfg.T]) if cfg.has_shared else 0)
    return {"rows_per_expert": {"min": int(counts.min()), "median": float(np.median(counts)),
                                "max": int(counts.max())},
            "eta": float(loads.mean() / loads.max()) if loads.max() > 0 else 1.0,
            "drop_fraction": float(1.0 - kept.sum() / max(cfg.A, 1)),
            "padding_fraction": float(1.0 - rows_kept / max(rows_tiled, 1)),
            "rows_kept": rows_kept, "rows_computed": rows_tiled,
            "capacity_padding_rows": int(cfg.R - kept.sum()) if cfg.capacity else 0}


class _L2Flush:
    """Evicts L2 between timed steps: a 512 MiB write (four times the 126 MB L2),
    then a 256 MiB read, so that the write's dirty lines go back to HBM before
    the next timed event rather than during the first timed kernel."""

    def __init__(self, dev):
        self.w = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(256 << 20, dtype=torch.uint8, device=dev)
        self.sink = torch.zeros((), dtype=torch.int64, device=dev)

    def __call__(self):
        self.w.zero_()
        torch.sum(self.r, dim=0, dtype=torch.int64, out=self.sink)


def _time_extras(m, layer, c, cfg, x, st, flush, counts, pk, reps):
    """Calls outside the layer step, timed alone with CUDA events (L2 flushed
    before each): the FP8 dispatch pair and the load-balancing kernels, then the
    layer's backward."""
    dev = x.device

    def timed(fn):
        out = []
        for _ in range(reps + 1):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(st)
            fn()
            b.record(st)
            out.append((a, b))
        torch.cuda.synchronize(dev)
        return float(np.mean([a.elapsed_time(b) for a, b in out[1:]]))

    A, d = cfg.A, cfg.d
    out = {}
    # the short, latency-bound calls first, after a quarter second idle: timed
    # right after the e2e legs and the backward (tens to hundreds of ms of dense
    # GEMMs) they ran at a power-capped clock (Mixtral-shaped FP8 receive 34.5
    # against 27.2 us alone)
    send_fp8 = torch.empty(A, d, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize(dev)
    time.sleep(0.25)
    out = _time_fp8_and_balance(m, layer, c, cfg, x, st, flush, counts, pk, reps, timed, out,
                                send_fp8)
    del send_fp8
    if not layer.gather:
        out.update(_time_combine_epilogue(m, layer, c, cfg, x, counts, timed))
    # backward of the layer (routing fixed), on the forward's buffers
    if not layer.gather:
        out.update(_time_backward(m, layer, c, cfg, x, st, flush, counts, pk, reps))
    return out


def _time_combine_epilogue(m, layer, c, cfg, x, counts, timed):
    """The grouped FFN with the combine in GEMM 2's epilogue (bf16 reductions
    into y, no y_sorted) against the two calls it replaces, each timed alone
    the same way."""
    xs = x if cfg.has_shared else None
    y_f = torch.empty_like(layer.y)
    fused = timed(lambda: m.moe_grouped_ffn_combine(c, layer.x_sorted, xs, layer.counts,
                                                    layer.offsets, layer.W13, layer.W2, layer.h,
                                                    layer.order, layer.topk_gate, y_f, layer.ws))

    def unfused():
        m.moe_grouped_ffn(c, layer.x_sorted, xs, layer.counts, layer.offsets, layer.W13,
                          layer.W2, layer.h, layer.y_sorted, layer.ws)
        m.moe_combine(c, layer.y_sorted, layer.inv, layer.topk_gate, layer.y)
    pair = timed(unfused)
    kept = int(np.minimum(counts, cfg.capacity).sum()) if cfg.capacity else cfg.A
    rows = kept + (cfg.T if cfg.has_shared else 0)
    flops = 6.0 * cfg.d * cfg.f * rows
    return {"ffn_combine_fused": {"ms": fused, "tflops": flops / (fused * 1e-3) / 1e12,
                                  "unfused_ffn_then_combine_ms": pair,
                                  "tiles": "one-SM (the epilogue exists there only)"}}


def _time_backward(m, layer, c, cfg, x, st, flush, counts, pk, reps):
    """The three backward calls after a fresh forward, timed per call."""
    dev = x.device
    A, d = cfg.A, cfg.d
    out = {}
    layer.forward(x)
    gen = torch.Generator(device=dev).manual_seed(77)
    dy = torch.randn(cfg.T, d, generator=gen, device=dev).to(torch.bfloat16)
    layer.backward(x, dy)
    # the training forward keeps GEMM 1's pre-activations: the timed backward reads them
    g1 = torch.empty(layer.h.shape[0], 2 * cfg.f, dtype=torch.bfloat16, device=dev)
    m.moe_grouped_ffn_train(c, layer.x_sorted, x if c.has_shared else None, layer.counts,
                            layer.offsets, layer.W13, layer.W2, layer.h, layer.y_sorted, g1,
                            layer.ws)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    per = []
    for _ in range(reps):
        flush()
        ev[0].record(st)
        m.moe_combine_backward(c, dy, layer.y_sorted, layer.inv, layer.topk_gate, layer.d_o,
                               layer.dgate)
        ev[1].record(st)
        m.moe_grouped_ffn_backward(c, layer.x_sorted, x if c.has_shared else None, layer.counts,
                                   layer.offsets, layer.W13, layer.W13t, layer.W2t, layer.h,
                                   g1, layer.d_o, layer.dx_sorted, layer.dW13, layer.dW2,
                                   layer.bws, layer.ws)
        ev[2].record(st)
        m.moe_permute_backward(c, layer.dx_sorted, layer.inv, layer.dx)
        ev[3].record(st)
        torch.cuda.synchronize(dev)
        per.append([ev[i].elapsed_time(ev[i + 1]) for i in range(3)])
    per = np.array(per).mean(axis=0)
    kept = int(np.minimum(counts, cfg.capacity).sum()) if cfg.capacity else A
    rows_ffn = kept + (cfg.T if cfg.has_shared else 0)
    bw_flops = 12.0 * d * cfg.f * rows_ffn      # dh, dx (dgrad) + dW2, dW13 (wgrad)
    tf = bw_flops / (per[1] * 1e-3) / 1e12
    out["backward"] = {"ms": float(per.sum()), "combine_backward_ms": float(per[0]),
                       "grouped_ffn_backward_ms": float(per[1]),
                       "permute_backward_ms": float(per[2]),
                       "ffn_backward_tflops": tf,
                       "ffn_backward_frac_bf16_sustained": tf / (pk["bf16_tflops_sustained"]
                                                                 or pk["bf16_tflops"]),
                       "flops_counted": "12*d*f per kept row (dh, dx, dW2, dW13; GEMM 1's "
                                        "output kept by the training forward)"}
    return out


def _time_fp8_and_balance(m, layer, c, cfg, x, st, flush, counts, pk, reps, timed, out,
                          send_fp8):
    dev = x.device
    A, d = cfg.A, cfg.d
    send_scale = torch.empty(A, dtype=torch.float32, device=dev)
    ms_pack = timed(lambda: m.moe_ep_layout_fp8(c, layer.topk_idx, layer.offsets, layer.inv,
                                                layer.count_mat, layer.send_off, layer.recv_off,
                                                layer.send_idx, x, send_fp8, send_scale,
                                                layer.ws))
    ms_recv = timed(lambda: m.moe_dispatch_recv_fp8(c, send_fp8, send_scale, layer.send_idx,
                                                    layer.inv, layer.x_sorted))
    kept = int(np.minimum(counts, cfg.capacity).sum()) if cfg.capacity else A
    b_pack = cfg.T * d * 2 + A * d + 4 * A + 16 * A
    b_recv = A * d + 4 * A + 8 * A + kept * d * 2
    gbs = lambda b, ms: b / (ms * 1e-3) / 1e9  # noqa: E731
    out["ep_layout_fp8"] = {"ms": ms_pack, "gbs": gbs(b_pack, ms_pack),
                            "frac_hbm": gbs(b_pack, ms_pack) / pk["hbm_gbs"]}
    out["dispatch_recv_fp8"] = {"ms": ms_recv, "gbs": gbs(b_recv, ms_recv),
                                "frac_hbm": gbs(b_recv, ms_recv) / pk["hbm_gbs"]}
    del send_fp8
    bias = torch.zeros(cfg.E, dtype=torch.float32, device=dev)
    out["bias_update"] = {"ms": timed(lambda: m.moe_bias_update(c, layer.counts, 1e-4, bias))}
    slots = cfg.E // cfg.n_ep + 1
    i32 = dict(dtype=torch.int32, device=dev)
    copies, coff = torch.empty(cfg.E, **i32), torch.empty(cfg.E, **i32)
    crank = torch.empty(cfg.n_ep * slots, **i32)
    sexp = torch.empty(cfg.n_ep, slots, **i32)
    rload = torch.empty(cfg.n_ep, dtype=torch.float64, device=dev)
    out["eplb_plan"] = {"ms": timed(lambda: m.moe_eplb_plan(c, layer.counts, slots, copies, coff,
                                                            crank, sexp, rload)),
                        "slots_per_rank": slots}
    dest = torch.empty(A, **i32)
    Cm = torch.empty(cfg.n_ep, cfg.n_ep, **i32)
    out["eplb_dispatch"] = {"ms": timed(lambda: m.moe_eplb_dispatch(
        c, layer.topk_idx, layer.counts, layer.offsets, layer.inv, copies, coff, crank, dest, Cm))}
    return out


def _kernel_source_digest():
    """sha1 over the sources of the grouped GEMMs (both kernels and the PTX wrappers)."""
    import hashlib
    h = hashlib.sha1()
    for rel in ("expert_token_dispatch_moe_b300/csrc/grouped_ffn.cu",
                "expert_token_dispatch_moe_b300/csrc/grouped_pair.cu",
                "expert_token_dispatch_moe_b300/csrc/common.cuh"):
        with open(os.path.join(ROOT, rel), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def _profiled_traffic(cfg):
    """DRAM bytes (read + write) of the grouped GEMM launches of one step, from
    the committed ncu summary of this workload (profiles/grouped_gemm_<name>.md,
    line 'traffic_bytes_per_step: <bytes> source_sha1: <digest>').  None when
    there is no summary or the kernel source changed since it was captured."""
    path = os.path.join(ROOT, "profiles", f"grouped_gemm_{cfg.name}.md")
    if not os.path.exists(path):
        return None
    for ln in open(path):
        if ln.startswith("traffic_bytes_per_step:"):
            parts = ln.split()
            if len(parts) >= 4 and parts[3] == _kernel_source_digest():
                return float(parts[1])
    return None


def _ffn_bytes(cfg, counts_np):
    """Algorithmic DRAM bytes of the two grouped GEMMs: the weights of every
    expert that received rows (and the shared expert) once, A rows read once, h
    written and read once, y_sorted written once."""
    kept = np.minimum(counts_np, cfg.capacity) if cfg.capacity else counts_np
    touched = int((kept > 0).sum()) + (1 if cfg.has_shared else 0)
    rows = int(kept.sum()) + (cfg.T if cfg.has_shared else 0)
    w = touched * 3 * cfg.d * cfg.f * 2
    return w + rows * cfg.d * 2 * 2 + rows * cfg.f * 2 * 2


PEAK_RULE = ("burst bf16 peak, unless the timed region lasted at least 1 s with sw_power_cap "
             "active in more than half of its clock samples and the median SM clock below the "
             "maximum: then the sustained (power-capped) bf16 peak")


def _tensor_peak(pk, clocks, timed_s):
    """The bf16 denominator for a kernel timed in this run, by PEAK_RULE: the
    sustained peak was measured over seconds of back-to-back GEMMs at the
    power limit, so it applies only to a timed region that long that also ran
    capped and below the top clock."""
    c = clocks or {}
    capped = (timed_s >= 1.0 and c.get("power_cap_share", 0.0) > 0.5
              and c.get("sm_mhz") is not None and c.get("sm_max_mhz") is not None
              and c["sm_mhz"] < c["sm_max_mhz"])
    if capped and pk["bf16_tflops_sustained"]:
        return pk["bf16_tflops_sustained"], pk["source"] + " sustained"
    return pk["bf16_tflops"], pk["source"] + " burst"


def _roofline(cfg, ffn_ms, ffn_flops, ffn_bytes, pk, clocks, timed_s):
    """The dominant kernel (both grouped GEMM launches of a step) against the
    roofline that bounds it: the bf16 peak when its FLOPs take longer than its
    bytes at the measured copy bandwidth, else HBM.  The bf16 denominator
    follows PEAK_RULE from this run's own clock samples; both fractions are
    reported."""
    peak_tf, src = _tensor_peak(pk, clocks, timed_s)
    t_flops = ffn_flops / (peak_tf * 1e12)
    t_bytes = ffn_bytes / (pk["hbm_gbs"] * 1e9)
    tflops = ffn_flops / (ffn_ms * 1e-3) / 1e12
    import expert_token_dispatch_moe_b300 as m
    kname = "grouped_pair_kernel" if m.moe_ffn_pair_tiles(m.MoeCfg.from_layer(cfg)) \
        else "grouped_gemm_kernel"
    base = {"kernel": f"{kname} (GEMM 1 + GEMM 2 of one step)",
            "traffic": _profiled_traffic(cfg), "algorithmic_bytes": ffn_bytes,
            "algorithmic_flops": ffn_flops}
    if t_flops >= t_bytes:
        base.update({"bound": "tensor", "achieved": tflops, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": tflops / peak_tf, "peak_source": src, "peak_rule": PEAK_RULE,
                     "frac_of_burst_peak": tflops / pk["bf16_tflops"],
                     "frac_of_sustained_peak": (tflops / pk["bf16_tflops_sustained"]
                                                if pk["bf16_tflops_sustained"] else None)})
    else:
        gbs = ffn_bytes / (ffn_ms * 1e-3) / 1e9
        base.update({"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / pk["hbm_gbs"], "peak_source": pk["source"] + " copy",
                     "tflops": tflops, "frac_of_burst_peak": tflops / pk["bf16_tflops"],
                     "frac_of_sustained_peak": (tflops / pk["bf16_tflops_sustained"]
                                                if pk["bf16_tflops_sustained"] else None)})
    return base


def run_ours(args, cfg):
    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    import expert_token_dispatch_moe_b300 as m

    x = synth.make_x(cfg, device=dev, seed=synth.DATA_SEED + rank)
    W_r, lbias = synth.make_router(cfg, device=dev)
    W1, W3, W2 = synth.make_expert_weights(cfg, device=dev)
    gather = args.path == "gather"
    layer = m.MoELayer(cfg, W1, W3, W2, W_r=W_r, logit_bias=lbias, device=dev, gather=gather)
    del W1, W3
    torch.cuda.empty_cache()
    c = layer.cfg
    st = torch.cuda.current_stream(dev)
    flush = _L2Flush(dev)

    names = ["router", "route", "permute", "ep_layout", "grouped_ffn", "combine"]

    def step(ev):
        ev[0].record(st)
        m.moe_router_logits(c, x, layer.W_r, layer.W_r_split, layer.logit_bias, layer.scores,
                            layer.ws)
        ev[1].record(st)
        m.moe_route(c, layer.scores, None, layer.topk_idx, layer.topk_gate)
        ev[2].record(st)
        m.moe_permute(c, None if gather else x, layer.topk_idx, layer.counts, layer.offsets,
                      layer.order, layer.inv, None if gather else layer.x_sorted, layer.ws)
        ev[3].record(st)
        m.moe_ep_layout(c, layer.topk_idx, layer.offsets, layer.inv, layer.count_mat,
                        layer.send_off, layer.recv_off, layer.send_idx, x, layer.send_buf, layer.ws)
        ev[4].record(st)
        if gather:
            m.moe_grouped_ffn_gather(c, x, layer.order, layer.counts, layer.offsets, layer.W13,
                                     layer.W2, layer.h, layer.y_sorted, layer.ws)
        else:
            m.moe_grouped_ffn(c, layer.x_sorted, x if c.has_shared else None, layer.counts,
                              layer.offsets, layer.W13, layer.W2, layer.h, layer.y_sorted,
                              layer.ws)
        ev[5].record(st)
        m.moe_combine(c, layer.y_sorted, layer.inv, layer.topk_gate, layer.y)
        ev[6].record(st)

    # launches per step, from the library's own accounting
    layer.forward(x)
    launches_per_step = layer.launches_per_forward
    for _ in range(args.warmup):
        flush()
        step([torch.cuda.Event(enable_timing=True) for _ in range(7)])
    torch.cuda.synchronize(dev)
    status = m.moe_get_device_status(layer.ws)
    if status != 0:
        raise RuntimeError(f"device status {status} after warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(args.steps)]
    clocks = _Clocks(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    t0 = time.perf_counter()
    for i in range(args.steps):
        flush()
        step(evs[i])
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t0
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    per = np.array([[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(6)]
                    for i in range(args.steps)])  # ms
    step_ms = float(per.sum(1).mean())
    step_ms = _max_over_ranks(step_ms, dev, world)
    status = m.moe_get_device_status(layer.ws)
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed steps")

    # end to end through the library's host call (moe_layer_forward_host): pinned
    # host x in and y out, one copy per direction per batch on copy streams, the
    # forward issued from C.  Serial: one batch per call, L2 flushed between
    # steps, so each step's copies and compute run back to back.
    x_host = x.cpu().pin_memory()
    y_host = torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16).pin_memory()
    e_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(args.steps)]
    for _ in range(2):
        layer.forward_host_c([x_host], [y_host])
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        flush()
        e_evs[i][0].record(st)
        layer.forward_host_c([x_host], [y_host])
        e_evs[i][1].record(st)
    torch.cuda.synchronize(dev)
    e2e_serial_ms = float(np.mean([a.elapsed_time(b) for a, b in e_evs]))

    # streamed: all `steps` batches in one call, each batch's host->device copy
    # and the previous batch's device->host copy overlapping compute; the whole
    # run is timed, so every step's copies are inside the region.  No flush
    # between steps here: the weights a step streams (>= 1 GB on the large
    # workloads) are far larger than L2.
    x_hosts, y_hosts = [x_host] * args.steps, [y_host] * args.steps
    layer.forward_host_c(x_hosts[:3], y_hosts[:3])
    torch.cuda.synchronize(dev)
    flush()
    s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s_ev.record(st)
    layer.forward_host_c(x_hosts, y_hosts)
    e_ev.record(st)
    torch.cuda.synchronize(dev)
    e2e_ms = s_ev.elapsed_time(e_ev) / args.steps
    e2e_ms = _max_over_ranks(e2e_ms, dev, world)

    counts = layer.counts.cpu().numpy()
    alg = _algorithmic(cfg, counts, gather)
    pk = _peaks()
    extra = _time_extras(m, layer, c, cfg, x, st, flush, counts, pk, reps=max(3, min(20, args.steps)))
    kt = {n: float(per[:, j].mean()) for j, n in enumerate(names)}  # ms per call
    ffn_tflops = alg["ffn_flops"] / (kt["grouped_ffn"] * 1e-3) / 1e12
    gbs = lambda b, ms: b / (ms * 1e-3) / 1e9  # noqa: E731
    kernels = {
        "grouped_ffn": {"ms": kt["grouped_ffn"], "tflops": ffn_tflops,
                        "frac_bf16_peak": ffn_tflops / pk["bf16_tflops"],
                        "frac_bf16_sustained": (ffn_tflops / pk["bf16_tflops_sustained"]
                                                if pk["bf16_tflops_sustained"] else None)},
        "router": {"ms": kt["router"], "gbs": gbs(alg["router_bytes"], kt["router"])},
        "route": {"ms": kt["route"], "gbs": gbs(alg["route_bytes"], kt["route"])},
        "permute": {"ms": kt["permute"], "gbs": gbs(alg["permute_bytes"], kt["permute"]),
                    "frac_hbm": gbs(alg["permute_bytes"], kt["permute"]) / pk["hbm_gbs"]},
        "ep_layout": {"ms": kt["ep_layout"], "gbs": gbs(alg["layout_bytes"], kt["ep_layout"]),
                      "frac_hbm": gbs(alg["layout_bytes"], kt["ep_layout"]) / pk["hbm_gbs"]},
        "combine": {"ms": kt["combine"], "gbs": gbs(alg["combine_bytes"], kt["combine"]),
                    "frac_hbm": gbs(alg["combine_bytes"], kt["combine"]) / pk["hbm_gbs"]},
    }
    kernels.update(extra)
    res = {
        "metric": METRIC,
        "value": cfg.T * world / (step_ms * 1e-3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": step_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded: x~N(0,1), expert weights~N(0,1/d), W_r~N(0,1/d) fp32)",
        "config": {"workload": _workload(cfg), "tokens_per_gpu": cfg.T, "path": args.path,
                   "l2": "flushed between timed steps (512 MiB write, then a 256 MiB read that writes the dirty lines back; outside the timed events)",
                   "parallelism": f"{world} independent replica(s)"},
        "e2e": {"value": cfg.T * world / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": cfg.T * cfg.d * 2, "d2h_bytes_per_step": cfg.T * cfg.d * 2,
                "ms_per_step": e2e_ms,
                "how": "moe_layer_forward_host (C ABI) over all steps: pinned host x in, y "
                       "out, one cudaMemcpyAsync per direction per batch on copy streams "
                       "overlapping compute, two device buffers per side",
                "serial": {"value": cfg.T * world / (e2e_serial_ms * 1e-3),
                           "ms_per_step": e2e_serial_ms,
                           "how": "moe_layer_forward_host with one batch per call (copy in, "
                                  "layer, copy out), L2 flushed between steps"}},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": _roofline(cfg, kt["grouped_ffn"], alg["ffn_flops"], _ffn_bytes(cfg, counts),
                              pk, clk, wall),
        "kernels": kernels,
        "layout": layout_metrics(cfg, counts, layer.count_mat.cpu().numpy()),
        "wall_s": wall,
    }
    if clk:
        res["clocks"] = clk
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(cfg, x, W_r, lbias, layer)
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(res), flush=True)


def _cores():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count()


# The oracle's timed sample per workload: (tokens in the sub-batch, routed experts
# whose rows the expert FFN computes).  Routing, permutation, EP layout and
# combine run on the whole sub-batch; the expert FFN on the complete segments of
# a seeded subset of the experts.  Sized so that one sample takes about a
# second on 16 host cores: a Mixtral expert's 128 rows of the 512-token batch
# cost 45 GFLOP in fp64, a DeepSeek-V3-shaped expert's 16 rows stream 350 MB of
# fp64 weights.
ORACLE_SAMPLE = {"tiny": (1024, 8), "mixtral": (512, 2), "dsv3": (512, 16),
                 "dsv3_decode": (128, 16), "skew": (4096, 16)}


class OracleSample:
    """One bounded sample of the workload on the oracle, as it stands: the
    first n tokens as one complete batch through the oracle's steps in the
    pages' order (router logits, expert choice and gates, permutation, EP
    layout, SwiGLU experts, combine), with the expert FFN computed on the rows
    of a seeded subset S of the routed experts.  The weights of S are upcast to
    fp64 once, before any timing, so the oracle's own upcast is a no-op and its
    cost is linear in the rows.  The full step is estimated by scaling the FFN
    time by (rows of the batch, shared rows included) / (rows of S), then the
    whole batch by T / n."""

    def __init__(self, cfg, x, W_r, lbias, expert_weights):
        """x, W_r, lbias: torch tensors (any device); expert_weights(ids) ->
        (W1, W3, W2) torch tensors of those experts, [len(ids), ...]."""
        import oracle
        self.oracle = oracle
        n, m = ORACLE_SAMPLE.get(cfg.name, (min(cfg.T, 512), min(cfg.E, 16)))
        n = min(n, cfg.T)
        m = min(m, cfg.E)
        self.cfg = cfg
        # the sub-batch keeps the workload's capacity factor (rows per expert scale with T)
        cap = max(1, math.ceil(cfg.capacity * n / cfg.T)) if cfg.capacity else 0
        self.sub = cfg.with_(T=n, n_ep=math.gcd(n, math.gcd(cfg.n_ep, cfg.E)), capacity=cap)
        self.x = x[:n].float().cpu().numpy()
        self.W_r = W_r.cpu().numpy()
        self.lbias = None if lbias is None else lbias.cpu().numpy()
        rng = np.random.default_rng(11)
        self.S = np.sort(rng.choice(cfg.E, m, replace=False))
        W1, W3, W2 = expert_weights([int(e) for e in self.S])
        self.W = {}
        for i, e in enumerate(self.S):
            self.W[int(e)] = tuple(np.asarray(w[i].float().cpu().numpy(), np.float64)
                                   for w in (W1, W3, W2))
        self.n, self.m = n, m

    def run(self):
        """One sample.  Returns (measured seconds, estimated seconds of the full
        step, rows of S, rows of the sub-batch)."""
        o, sub = self.oracle, self.sub
        W = self.W
        t0 = time.perf_counter()
        l = o.router_logits(self.x, self.W_r, self.lbias)
        s = (o.sigmoid(l) if sub.score_fn == "sigmoid" else l).astype(np.float32)
        idx = o.select_experts(s, sub.k, None, sub.n_groups, sub.topk_groups)
        gates = o.gate_weights(s, idx, sub.score_fn, sub.norm_topk)
        perm = o.permute(idx, sub.E, sub.capacity)
        o.ep_layout(idx, perm["inv"], sub.E, sub.n_ep, sub.T)
        t1 = time.perf_counter()
        segs = [np.arange(int(perm["offsets"][e]), int(perm["offsets"][e] + perm["kept"][e]))
                for e in W]
        rows = np.concatenate(segs) if segs else np.zeros(0, np.int64)
        view = lambda j: {e: W[e][j] for e in W}  # noqa: E731
        out = o.expert_outputs(self.x, perm, sub.k, view(0), view(1), view(2), rows=rows)
        t2 = time.perf_counter()
        o.combine(out, perm, sub.k, gates, sub.T)
        t3 = time.perf_counter()
        ffn = t2 - t1
        rows_all = int(perm["kept"].sum()) + (sub.T if sub.has_shared else 0)
        est = ((t1 - t0) + (t3 - t2) + ffn * rows_all / max(rows.size, 1)) * self.cfg.T / sub.T
        return t3 - t0, est, int(rows.size), rows_all

    def describe(self, rows_s, rows_all):
        return (f"first {self.n} tokens as one batch (router, routing, permutation, EP layout, "
                f"combine) with the expert FFN on the complete segments of {self.m} seeded "
                f"experts ({rows_s} of the batch's {rows_all} rows), fp64 weights of those "
                f"experts upcast once before timing; the full {self.cfg.T}-token step is "
                f"estimated as (batch time with the FFN scaled by rows) x {self.cfg.T}/{self.n}")


def cpu_baseline(cfg, x, W_r, lbias, layer, reps=3, min_s=10.0, max_reps=40):
    """The oracle, as it stands, on the bounded sample of OracleSample (the
    same procedure as --impl reference): after one warm run, at least `reps`
    runs and more until about `min_s` seconds of host work (at most `max_reps`
    runs); the median of the runs."""
    def weights(ids):
        W13, W2 = layer.W13, layer.W2
        n, f2, d = W13.shape
        blk = W13[ids].view(len(ids), f2 // 256, 2, 128, d)  # undo the 128-row interleave
        return (blk[:, :, 0].reshape(len(ids), f2 // 2, d),
                blk[:, :, 1].reshape(len(ids), f2 // 2, d), W2[ids])
    samp = OracleSample(cfg, x, W_r, lbias, weights)
    samp.run()  # warm
    runs, spent = [], 0.0
    while len(runs) < reps or (spent < min_s and len(runs) < max_reps):
        runs.append(samp.run())
        spent += runs[-1][0]
    meas = statistics.median(r[0] for r in runs)
    est = statistics.median(r[1] for r in runs)
    return {"value": cfg.T / est, "unit": "tokens/s", "cores": _cores(), "kind": "oracle",
            "sample": samp.describe(runs[0][2], runs[0][3]), "sample_s": meas,
            "sample_tokens": samp.n, "estimated_step_s": est, "sample_runs": len(runs),
            "host_s": spent}


def run_reference(args, cfg):
    world, rank, _ = _dist()
    if rank != 0:
        return
    x = synth.make_x(cfg)
    W_r, lbias = synth.make_router(cfg)
    samp = OracleSample(cfg, x, W_r, lbias,
                        lambda ids: synth.make_expert_weights(cfg, experts=ids))
    for _ in range(args.warmup):
        samp.run()
    runs = [samp.run() for _ in range(args.steps)]
    meas = float(np.mean([r[0] for r in runs]))
    est = float(np.mean([r[1] for r in runs]))
    v = cfg.T / est
    res = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": meas * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": _workload(cfg), "tokens_per_gpu": cfg.T,
                   "parallelism": "host cores (oracle)"},
        "timing": {"ms_per_step": "measured time of one sample step (the timed region is "
                                  "steps x this)",
                   "estimated_full_step_ms": est * 1e3,
                   "value": "T / estimated full step"},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": _cores(), "kind": "oracle",
                         "sample": samp.describe(runs[0][2], runs[0][3]),
                         "sample_s": meas, "sample_tokens": samp.n, "estimated_step_s": est},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(res), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="dsv3", choices=sorted(synth.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--path", default="rows", choices=["rows", "gather"],
                    help="rows: the permute writes x_sorted and GEMM 1 reads it; gather: the "
                         "permute computes indices only and GEMM 1 gathers token rows itself")
    ap.add_argument("--override", default="",
                    help="comma-separated field=value changes to the workload, e.g. "
                         "T=1024,E=32,n_ep=8 (a reduced case of the same shape for profiling)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    cfg = synth.CONFIGS[args.config]
    if args.override:
        kw = {}
        for item in args.override.split(","):
            key, val = item.split("=")
            kw[key.strip()] = type(getattr(cfg, key.strip()))(val)
        cfg = cfg.with_(name=cfg.name + "[" + args.override + "]", **kw)
    if args.impl == "reference":
        run_reference(args, cfg)
    else:
        run_ours(args, cfg)


if __name__ == "__main__":
    main()
