"""Benchmark of the GB300 quantized attention path.

One step = the whole dense path over the 37,810-token, 24-head video-DiT
self-attention workload (B=1, H=24, Nq=Nk=37,810, d=128, Q/K INT8 per
128-token blocks, FP8 V): sage_quantize_qkv (K smoothing, Q/K INT8 codes as
their exact fp16 images, V FP8 codes; three launches) + sage_attn_fwd_f16
(the attention kernel), inputs already resident in HBM.  The metric is
effective TFLOP/s (4 * Nq * Nk * d * H per step); ms per step is reported
beside it.

Also measured in the same run (JSON keys, not extra lines):
  * per-call times of the two calls (CUDA events around each call inside the
    timed steps), the roofline of the attention kernel against the measured
    peaks and against the tensor core's own per-clock rates (the library's
    rate probe), and the same path as three separate entry points;
  * per-config results for the five workloads (GPU time, CPU oracle time,
    whole-head parity against the oracle);
  * int8kv_prompt_attn on the 32K x 1024 and 64K x 512 int8 KV-cache chunks;
  * e2e: the same step through the public API with pinned host buffers
    (sage_attention_host: host->device copy of Q, K, V and device->host copy
    of the output inside the timed region, overlapped with the kernels of the
    previous group of heads);
  * cpu_baseline: the CPU oracle on a bounded sample of the workload.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun the global batch holds one 24-head problem per rank and the
24 * N independent heads are split over the ranks by the library's
sage_shard_range (24 heads each, no collective on the data path: weak
scaling); rank 0 prints the line with the maximum time over ranks.
"""

from __future__ import annotations

import argparse
import gc
import hashlib
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

import synth  # noqa: E402

METRIC = "quantized attention fwd effective TFLOPS (4*Nq*Nk*d*H), video-DiT 37,810-token self-attention"
UNIT = "TFLOP/s"
WORKLOAD = "videodit_b1h24n37810"

# DRAM bytes (read + write) per launch of the attention kernel, from one ncu
# capture of the 24-head, 16,384-token case (the fp16 images exceed L2 there):
# 251.9 MB read + 72.3 MB written, scaled by 37,810 / 16,384 (every head's
# inputs are read once, so the bytes grow with heads x tokens); and the kernel's
# tensor-pipe activity from the full ncu capture of the 8,192-token case.  Both
# hold for the kernel source with this sha256 prefix and are None once the
# source has changed.
TRAFFIC = {"sha256_prefix": "588cb0f979b58405", "bytes": (251.9e6 + 72.3e6) * 37810 / 16384,
           "tensor_pipe_active": 0.511}
# algorithmic bytes of one attention launch at the full workload: Q, K, V codes
# (1 byte per element) and the bf16 output
ATTN_METHOD_BYTES = 24 * 37810 * 128 * (1 + 1 + 1 + 2)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def cpu_model() -> str:
    """The host CPU's model as lscpu reports it (empty if unavailable)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
    except (OSError, subprocess.TimeoutExpired):
        return ""
    for line in out.splitlines():
        if line.strip().startswith("Model name:"):
            return line.split(":", 1)[1].strip()
    return ""


def current_sms(dev) -> int:
    import torch

    return torch.cuda.get_device_properties(dev).multi_processor_count


def kernel_sha(name: str) -> str:
    p = os.path.join(ROOT, "quantized_attention_sage_gb300", "csrc", name)
    return hashlib.sha256(open(p, "rb").read()).hexdigest()


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append(parts)
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        loaded = [s for s, p in zip(sm, power) if p >= 0.5 * max(power)] if power else sm
        return {"sm_mhz": statistics.median(loaded or sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons, "samples": len(rows),
                "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample
# ---------------------------------------------------------------------------

_ORACLE_INPUTS = {}


def kv_cache_on_device(qas, torch, y: dict, dev):
    """Queries and the int8 KV cache on the device: the cache is written from the
    workload's fp32 rows by the library's cache writer (outside any timed region)."""
    q = torch.from_numpy(y["q"].view(np.int16)).view(torch.bfloat16).to(dev)
    k = torch.from_numpy(y["k_raw"]).to(dev).permute(1, 0, 2)  # token-major view [Nk, Hkv, 128]
    v = torch.from_numpy(y["v_raw"]).to(dev).permute(1, 0, 2)
    hkv, nk, d = y["k_raw"].shape
    kc = torch.empty((hkv, nk, d), dtype=torch.int8, device=dev)
    vc = torch.empty_like(kc)
    ks = torch.empty((hkv, nk), dtype=torch.float16, device=dev)
    vs = torch.empty_like(ks)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    qas.int8kv_cache_write(k, v, kc, ks, vc, vs, 0, status=status)
    torch.cuda.synchronize(dev)
    assert status.item() == 0, "device status set by the cache writer"
    return q, kc, ks, vc, vs


def oracle_sample(target_s: float = 12.0):
    """Time the oracle on one head of the workload: its quantisation and the
    attention of a sample of query rows, scaled to the whole workload."""
    import oracle

    w = synth.dense_workload(WORKLOAD)
    if "head0" not in _ORACLE_INPUTS:
        _ORACLE_INPUTS["head0"] = synth.dense_inputs(w, heads=(0, 1))
    x = _ORACLE_INPUTS["head0"]
    q, k, v = x["q"][0, 0], x["k"][0, 0], x["v"][0, 0]
    t0 = time.perf_counter()
    mu = oracle.k_mean(k)
    qc, sq = oracle.quant_q(q, w.block)
    kc, sk = oracle.quant_k(k, w.block, mu)
    vct, sv = oracle.quant_v(v)
    t_quant = time.perf_counter() - t0
    rng = np.random.default_rng(3)
    rows_done, t_rows, threads = 0, 0.0, 1
    batch = 32
    while t_rows < target_s and rows_done < w.Nq:
        rows = rng.integers(0, w.Nq, batch).astype(np.int32)
        t1 = time.perf_counter()
        _, _, threads = oracle.sage_attn_rows(qc, sq, w.block, kc, sk, w.block, vct, sv, w.Nq, w.Nk, rows=rows)
        t_rows += time.perf_counter() - t1
        rows_done += batch
        if t_rows > 0 and rows_done == batch:
            batch = max(batch, int(batch * (target_s / 2) / t_rows))
    per_row = t_rows / rows_done
    est_s = w.B * w.H * (t_quant + per_row * w.Nq)
    return {"value": w.flops / est_s / 1e12, "unit": UNIT, "cores": int(threads), "kind": "oracle",
            "sample": (f"head 0 of {WORKLOAD}: quantisation of the head ({t_quant:.2f} s) and the "
                       f"attention of {rows_done} random query rows ({t_rows:.2f} s), scaled to "
                       f"24 heads x 37,810 rows"),
            "seconds": t_quant + t_rows, "est_full_seconds": est_s}


def per_clock_peak(probe: dict, sms: int, mhz: float) -> float:
    """Mixed TFLOP/s peak of the dense attention (equal FLOPs on kind::f16 and
    kind::f8f6f4) from the probe's MACs per SM per clock at `mhz`."""
    p16 = 2 * probe["f16_mac_per_clk_sm"] * sms * mhz * 1e6 / 1e12
    p8 = 2 * probe["f8_mac_per_clk_sm"] * sms * mhz * 1e6 / 1e12
    return 2.0 / (1.0 / p16 + 1.0 / p8)


def _pct(xs):
    xs = sorted(xs)
    at = lambda f: xs[int(round(f * (len(xs) - 1)))]  # noqa: E731
    return {"p10": at(0.1), "p50": at(0.5), "p90": at(0.9)}


def _per_call_ms(torch, fn, reps, stream):
    """CUDA-event time of each of `reps` calls (after 3 warm-up calls)."""
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    ev[0].record(stream)
    for i in range(reps):
        fn()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    return [ev[i].elapsed_time(ev[i + 1]) for i in range(reps)]


def _rel_l2(got, ref):
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def _bits_f64(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def _fp64_attention(q, k, v, sm_scale, visible=None):
    """Unquantised softmax(q k^T sm_scale) v in fp64; visible[i] = keys row i sees (causal)."""
    s = (q @ k.T) * sm_scale
    if visible is not None:
        s = np.where(np.arange(k.shape[0])[None, :] < visible[:, None], s, -np.inf)
    s -= s.max(axis=1, keepdims=True)
    p = np.exp(s)
    return (p @ v) / p.sum(axis=1, keepdims=True)


def per_config_results(qas, torch, dev, pk, peak_mixed, main):
    """The five configurations: GPU time (p10/p50/p90 of single calls), effective
    TFLOP/s and roofline fraction, the CPU oracle's time on the host cores, and
    parity of whole heads (whole kv-head groups) against the oracle, with the
    distance of the GPU result from unquantised fp64 attention."""
    import oracle

    stream = torch.cuda.current_stream()
    sms_scale = 1.0 / math.sqrt(128.0)
    res = []
    p16 = pk["bf16_tflops"]

    def dev_bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    # configs 1 and 2: the one-call dense path on small inputs (latency-bound)
    for w in synth.dense_workloads():
        if w.config not in (1, 2):
            continue
        x = synth.dense_inputs(w)
        q, k, v = dev_bf16(x["q"]), dev_bf16(x["k"]), dev_bf16(x["v"])
        out = torch.empty((w.B, w.H, w.Nq, 128), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(qas.lib().sage_attention_workspace(w.B, w.H, w.Nq, w.Nk), dtype=torch.uint8, device=dev)
        ms = _per_call_ms(torch, lambda: qas.sage_attention(q, k, v, w.block, w.block, out=out, workspace=ws), 30,
                          stream)
        got = out.float().cpu().numpy().astype(np.float64)[0]
        cpu, refs, threads = [], None, 1
        for _ in range(3):
            t0 = time.perf_counter()
            refs = [oracle.sage_head(x["q"][0, h], x["k"][0, h], x["v"][0, h], w.block, w.block) for h in range(w.H)]
            cpu.append((time.perf_counter() - t0) * 1e3)
            threads = refs[0]["threads"]
        ref = np.stack([_bits_f64(r["out_bf16"]) for r in refs])
        f64 = np.stack([_fp64_attention(_bits_f64(x["q"][0, h]), _bits_f64(x["k"][0, h]), _bits_f64(x["v"][0, h]),
                                        sms_scale) for h in range(w.H)])
        t = _pct(ms)
        res.append({"config": w.config, "workload": w.name, "gpu_ms": t, "call": "sage_attention (one call)",
                    "tflops": w.flops / (t["p50"] * 1e-3) / 1e12,
                    "roofline_frac": w.flops / (t["p50"] * 1e-3) / 1e12 / peak_mixed,
                    "cpu_oracle_ms": statistics.median(cpu), "cpu_cores": threads, "cpu_extrapolated": False,
                    "parity": {"rows": w.H * w.Nq, "max_abs": float(np.abs(got - ref).max()),
                               "rel_l2": _rel_l2(got, ref), "rel_l2_vs_fp64_unquantised": _rel_l2(got, f64)}})

    # config 3: timings of the main loop; one whole head against the oracle
    # (its time, x 24 heads, is the CPU figure)
    w = synth.dense_workload(WORKLOAD)
    h = 11
    x = synth.dense_inputs(w, heads=(h, h + 1))
    t0 = time.perf_counter()
    ref = oracle.sage_head(x["q"][0, 0], x["k"][0, 0], x["v"][0, 0], w.block, w.block)
    t_head = time.perf_counter() - t0
    got = main["dense_out"]()[0, h].float().cpu().numpy().astype(np.float64)
    refb = _bits_f64(ref["out_bf16"])
    rows = np.random.default_rng(9).choice(w.Nq, 1024, replace=False)
    f64 = _fp64_attention(_bits_f64(x["q"][0, 0][rows]), _bits_f64(x["k"][0, 0]), _bits_f64(x["v"][0, 0]), sms_scale)
    t = _pct(main["attn_ms"])
    res.append({"config": w.config, "workload": w.name, "gpu_ms": t, "call": "sage_attn_fwd_f16",
                "step_ms": _pct(main["step_ms"]), "tflops": w.flops / (t["p50"] * 1e-3) / 1e12,
                "roofline_frac": w.flops / (t["p50"] * 1e-3) / 1e12 / peak_mixed,
                "cpu_oracle_ms": t_head * w.H * 1e3, "cpu_cores": ref["threads"], "cpu_extrapolated": True,
                "cpu_note": f"one whole head (quantisation + all {w.Nq} rows) in {t_head:.1f} s, x {w.H} heads",
                "parity": {"rows": w.Nq, "head": h, "max_abs": float(np.abs(got - refb).max()),
                           "rel_l2": _rel_l2(got, refb), "rel_l2_vs_fp64_unquantised": _rel_l2(got[rows], f64),
                           "fp64_rows": int(rows.size)}})

    # configs 4 and 5: one whole kv-head group against the fp64 oracle (its
    # time, x Hkv groups, is the CPU figure); distance from fp64 attention over
    # the unquantised fp32 K/V rows of that group
    for name in ("prompt32k_q1024", "prompt64k_q512_outliers"):
        wk = synth.int8kv_workload(name)
        y = synth.int8kv_inputs(wk)
        tq, kc, ks, vc, vs = kv_cache_on_device(qas, torch, y, dev)
        o = torch.empty((wk.Nq, wk.Hq, 128), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(qas.lib().int8kv_prompt_attn_workspace(wk.Nq, wk.Hq, wk.Hkv, wk.Nk), dtype=torch.uint8,
                         device=dev)
        ms = _per_call_ms(torch, lambda: qas.int8kv_prompt_attn(tq, kc, ks, vc, vs, wk.q_pos0, out=o, workspace=ws),
                          20, stream)
        G = wk.Hq // wk.Hkv
        g = wk.Hkv - 1
        host = {"q": y["q"]}
        for key in ("k", "v"):
            codes, bits = oracle.cache_quantise(y[key + "_raw"])
            host[key], host[key + "_scale"] = codes, bits.view(np.float16)
        assert np.array_equal(kc.cpu().numpy(), host["k"]) and np.array_equal(vc.cpu().numpy(), host["v"])
        rr, hh = np.meshgrid(np.arange(wk.Nq), np.arange(g * G, (g + 1) * G), indexing="ij")
        rr, hh = rr.ravel(), hh.ravel()
        t0 = time.perf_counter()
        ref, threads = oracle.int8kv_rows(host["q"], host["k"], host["k_scale"], host["v"], host["v_scale"],
                                          wk.q_pos0, rr, hh)
        t_grp = time.perf_counter() - t0
        refb = oracle.bf16_value(oracle.f32_to_bf16(ref.astype(np.float32)))
        got = o[torch.as_tensor(rr).to(dev), torch.as_tensor(hh).to(dev)].float().cpu().numpy().astype(np.float64)
        f64 = np.concatenate([_fp64_attention(_bits_f64(y["q"][:, hd]), y["k_raw"][g].astype(np.float64),
                                              y["v_raw"][g].astype(np.float64), sms_scale,
                                              visible=wk.q_pos0 + np.arange(wk.Nq) + 1)
                              for hd in range(g * G, (g + 1) * G)])
        got_by_head = np.concatenate([got[hh == hd] for hd in range(g * G, (g + 1) * G)])
        t = _pct(ms)
        visible = 4 * wk.visible_pairs * 128 * wk.Hq
        res.append({"config": wk.config, "workload": name, "gpu_ms": t, "call": "int8kv_prompt_attn",
                    "tflops": wk.flops / (t["p50"] * 1e-3) / 1e12,
                    "tflops_causal": visible / (t["p50"] * 1e-3) / 1e12,
                    "roofline_frac": visible / (t["p50"] * 1e-3) / 1e12 / p16,
                    "cpu_oracle_ms": t_grp * wk.Hkv * 1e3, "cpu_cores": threads, "cpu_extrapolated": True,
                    "cpu_note": f"one whole kv group ({rr.size} rows) in {t_grp:.1f} s, x {wk.Hkv} groups",
                    "parity": {"rows": int(rr.size), "kv_group": g, "max_abs": float(np.abs(got - refb).max()),
                               "rel_l2": _rel_l2(got, refb),
                               "rel_l2_vs_fp64_unquantised": _rel_l2(got_by_head, f64)}})
        del tq, kc, ks, vc, vs, o, ws
    return res, {"value": w.flops / (t_head * w.H) / 1e12, "unit": UNIT, "cores": int(ref_threads(res)),
                 "kind": "oracle", "extrapolated": True,
                 "sample": (f"head {h} of {WORKLOAD}: quantisation and all {w.Nq} query rows "
                            f"({t_head:.1f} s), scaled to {w.H} heads")}


def ref_threads(res):
    return next(r["cpu_cores"] for r in res if r["config"] == 3)


def run_reference(args, rank):
    if rank != 0:
        return
    per_step = max(2.0, min(15.0, 60.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(per_step / 4)
    vals, secs = [], []
    last = None
    for _ in range(args.steps):
        last = oracle_sample(per_step)
        vals.append(last["value"])
        secs.append(last["est_full_seconds"])
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.median(secs) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded SplitMix64/Box-Muller, the workload's shapes)",
        "config": {"workload": WORKLOAD, "B": 1, "H": 24, "Nq": 37810, "Nk": 37810, "d": 128, "block": 128,
                   "note": ("CPU oracle (plain C, OpenMP) on a bounded sample, scaled to the workload: "
                            "ms_per_step is that extrapolation, not a timed run")},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": last["cores"], "kind": "oracle",
                         "sample": last["sample"], "extrapolated": True},
        "extrapolated": True,
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# multi-rank timing: every rank runs the whole workload on its own GPU (the
# (b, h) problems are independent, no collective on the data path); the job's
# time is the slowest rank's and the value counts the work of all ranks
# ---------------------------------------------------------------------------

def max_over_ranks(ms: float, dist=None, device=None) -> float:
    """The maximum of a per-rank time over all ranks (the value itself without a process group)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(ms)
    import torch

    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank: int, world: int, ms: float) -> float:
    """Aggregate throughput: the work of all ranks over the slowest rank's time."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args, rank, world):
    import torch

    import quantized_attention_sage_gb300 as qas

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist_mod

        dist_mod.init_process_group("nccl")
        dist = dist_mod
    qas.build()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()

    w = synth.dense_workload(WORKLOAD)
    # Multi-GPU: the global batch holds one 24-head problem per rank, i.e.
    # 24 * world independent heads, and sage_shard_range gives each rank its
    # contiguous share of them (24 heads: weak scaling, no collective on the
    # data path).  With one rank this is exactly the single-GPU workload.
    g = synth.DenseWorkload(WORKLOAD, w.config, 1, w.H * world, w.Nq, w.Nk, w.block)
    h0, h1 = qas.sage_shard_range(g.H, world, rank)
    assert h1 - h0 == w.H
    x = synth.dense_inputs(g, heads=(h0, h1))

    def to_pinned(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).pin_memory()

    hq, hk, hv = to_pinned(x["q"]), to_pinned(x["k"]), to_pinned(x["v"])
    q, k, v = hq.to(dev), hk.to(dev), hv.to(dev)
    B, H, N, D = q.shape
    bq = bk = w.block
    nb = -(-N // bq)
    qk = dict(q_codes=torch.empty((B, H, N, D), dtype=torch.int8, device=dev),
              q_scales=torch.empty((B, H, nb), dtype=torch.float32, device=dev),
              k_codes=torch.empty((B, H, N, D), dtype=torch.int8, device=dev),
              k_scales=torch.empty((B, H, nb), dtype=torch.float32, device=dev),
              k_mean=torch.empty((B, H, D), dtype=torch.float32, device=dev))
    vq = dict(v_codes=torch.empty((B, H, D, qas.nk_pad(N)), dtype=torch.uint8, device=dev),
              v_scales=torch.empty((B, H, D), dtype=torch.float32, device=dev))
    out = torch.empty((B, H, N, D), dtype=torch.bfloat16, device=dev)
    L = qas.lib()
    ws_qk = torch.empty(L.sage_quantize_qk_workspace(B, H, N), dtype=torch.uint8, device=dev)
    ws_v = torch.empty(L.sage_quantize_v_workspace(B, H, N), dtype=torch.uint8, device=dev)
    ws_a = torch.empty(L.sage_attn_fwd_workspace(B, H, N, N), dtype=torch.uint8, device=dev)
    ws_p = torch.empty(L.sage_quantize_qkv_workspace(B, H, N), dtype=torch.uint8, device=dev)
    prep = dict(q_codes=torch.empty((B, H, N, D), dtype=torch.float16, device=dev), q_scales=qk["q_scales"],
                k_codes=torch.empty((B, H, N, D), dtype=torch.float16, device=dev), k_scales=qk["k_scales"],
                k_mean=qk["k_mean"], v_codes=vq["v_codes"], v_scales=vq["v_scales"])
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    # One step = the whole dense path: the fused preparation (K smoothing, Q/K
    # INT8 codes written as their exact fp16 images, V FP8 codes: three
    # launches) and the attention kernel over the images.
    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        qas.sage_quantize_qkv(q, k, v, bq, bk, images=True, out=prep, workspace=ws_p)
        if ev is not None:
            ev[1].record(stream)
        qas.sage_attn_fwd_f16(prep, bq, bk, out=out, status=status)
        if ev is not None:
            ev[2].record(stream)

    # The same path as its three separate entry points (six quantizer launches,
    # two image passes inside sage_attn_fwd), timed for comparison.
    def three_calls(ev):
        ev[0].record(stream)
        qas.sage_quantize_qk(q, k, bq, bk, out=qk, workspace=ws_qk)
        ev[1].record(stream)
        qas.sage_quantize_v(v, out=vq, workspace=ws_v)
        ev[2].record(stream)
        qas.sage_attn_fwd(qk, vq, bq, bk, out=out, workspace=ws_a, status=status)
        ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert status.item() == 0, "device status set during warm-up"

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    ms_total = max_over_ranks(t_start.elapsed_time(t_end), dist, dev)
    assert status.item() == 0, "device status set during the timed steps"
    ms_step = ms_total / args.steps
    comp = {
        "sage_quantize_qkv_ms": statistics.mean(e[0].elapsed_time(e[1]) for e in evs),
        "sage_attn_fwd_f16_ms": statistics.mean(e[1].elapsed_time(e[2]) for e in evs),
    }
    step_each = [e[0].elapsed_time(e[2]) for e in evs]
    attn_each = [e[1].elapsed_time(e[2]) for e in evs]
    attn_ms = sorted(attn_each)
    comp["sage_attn_fwd_f16_ms_p10_p50_p90"] = [attn_ms[int(0.1 * (len(attn_ms) - 1))],
                                                attn_ms[int(0.5 * (len(attn_ms) - 1))],
                                                attn_ms[int(0.9 * (len(attn_ms) - 1))]]
    value = whole_job_tflops(w.flops, world, ms_step)
    # the three separate entry points, for comparison (after the timed steps)
    ev3 = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(5)]
    three_calls(ev3[0])
    torch.cuda.synchronize()
    for e in ev3:
        three_calls(e)
    torch.cuda.synchronize()
    assert status.item() == 0, "device status set by the three entry points"
    comp["three_entry_points"] = {
        "sage_quantize_qk_ms": statistics.mean(e[0].elapsed_time(e[1]) for e in ev3),
        "sage_quantize_v_ms": statistics.mean(e[1].elapsed_time(e[2]) for e in ev3),
        "sage_attn_fwd_ms": statistics.mean(e[2].elapsed_time(e[3]) for e in ev3),
        "step_ms": statistics.mean(e[0].elapsed_time(e[3]) for e in ev3)}

    # ---- end to end through the public API with pinned host buffers: sage_attention_host
    # copies groups of heads in and out on a copy stream while the previous group runs
    hout = torch.empty((B, H, N, D), dtype=torch.bfloat16).pin_memory()
    # about half a second of timed steps, so that the mean takes in proportion,
    # not all or nothing, the 40-80 ms stalls that sustained host-buffer calls
    # can show about every 0.5 s
    e2e_steps = max(2, min(5 * args.steps, 50))
    head_chunk = 6
    cstream, xstream = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ws_host = torch.empty(L.sage_attention_host_workspace(B, H, N, N, head_chunk), dtype=torch.uint8, device=dev)

    def e2e_step():
        qas.sage_attention_host(hq, hk, hv, hout, bq, bk, head_chunk=head_chunk, workspace=ws_host, status=status,
                                stream=cstream, copy_stream=xstream)

    for _ in range(max(3, args.warmup)):  # warm-up, as for the device steps
        e2e_step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps + 1)]
    enqueue_ms = []
    gc.collect()
    gc.disable()  # as timeit does: no collector pause inside the host-side enqueue of a step
    e0.record(cstream)
    step_ev[0].record(cstream)
    for i in range(e2e_steps):
        h0 = time.perf_counter()
        e2e_step()
        enqueue_ms.append((time.perf_counter() - h0) * 1e3)
        step_ev[i + 1].record(cstream)
    e1.record(cstream)
    torch.cuda.synchronize()
    gc.enable()
    assert status.item() == 0, "device status set during the e2e steps"
    ms_e2e = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dist, dev)
    per_step = [step_ev[i].elapsed_time(step_ev[i + 1]) for i in range(e2e_steps)]
    e2e = {"value": whole_job_tflops(w.flops, world, ms_e2e), "unit": UNIT, "ms_per_step": ms_e2e,
           "ms_median_step": statistics.median(per_step), "steps": e2e_steps,
           "ms_each_step": per_step, "host_enqueue_ms_each_step": enqueue_ms,
           "h2d_bytes_per_step": 3 * q.numel() * 2, "d2h_bytes_per_step": out.numel() * 2,
           "api": f"sage_attention_host, head_chunk={head_chunk}, pinned host buffers"}
    del ws_host

    # ---- causal dense attention with the row log-sum-exp, same workload and codes
    for _ in range(3):
        qas.sage_attn_fwd(qk, vq, bq, bk, out=out, workspace=ws_a, status=status, causal=True, return_lse=True)
    torch.cuda.synchronize()
    reps_c = max(5, args.steps // 2)
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    for _ in range(reps_c):
        qas.sage_attn_fwd(qk, vq, bq, bk, out=out, workspace=ws_a, status=status, causal=True, return_lse=True)
    c1.record(stream)
    torch.cuda.synchronize()
    assert status.item() == 0, "device status set in causal sage_attn_fwd"
    ms_c = c0.elapsed_time(c1) / reps_c
    visible = N * (N + 1) // 2  # query i sees keys 0..i
    causal = {"ms": ms_c, "tflops_visible": 4 * visible * D * H * B / (ms_c * 1e-3) / 1e12,
              "tflops_formula": w.flops / (ms_c * 1e-3) / 1e12, "lse": True}

    # ---- int8 KV-cache prompt attention
    kv = {}
    for name in ("prompt32k_q1024", "prompt64k_q512_outliers"):
        wk = synth.int8kv_workload(name)
        tq, kc, ks, vc, vs = kv_cache_on_device(qas, torch, synth.int8kv_inputs(wk), dev)
        o = torch.empty((wk.Nq, wk.Hq, 128), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(L.int8kv_prompt_attn_workspace(wk.Nq, wk.Hq, wk.Hkv, wk.Nk), dtype=torch.uint8, device=dev)
        for _ in range(3):
            qas.int8kv_prompt_attn(tq, kc, ks, vc, vs, wk.q_pos0, out=o, workspace=ws, status=status)
        torch.cuda.synchronize()
        reps = max(5, args.steps)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            qas.int8kv_prompt_attn(tq, kc, ks, vc, vs, wk.q_pos0, out=o, workspace=ws, status=status)
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / reps
        kv[name] = {"ms": ms, "tflops_formula": wk.flops / (ms * 1e-3) / 1e12,
                    "tflops_causal": 4 * wk.visible_pairs * 128 * wk.Hq / (ms * 1e-3) / 1e12,
                    "Nq": wk.Nq, "Nk": wk.Nk, "Hq": wk.Hq, "Hkv": wk.Hkv}
    assert status.item() == 0, "device status set in int8kv_prompt_attn"
    # ---- int8 KV-cache writer: the whole 32K cache of the prompt chunk from bf16 rows
    wk = synth.int8kv_workload("prompt32k_q1024")
    gen = torch.Generator(device=dev)
    gen.manual_seed(synth.seed_for(wk.config, synth.T_K))
    kr = torch.randn((wk.Nk, wk.Hkv, 128), generator=gen, device=dev).to(torch.bfloat16)
    vr = torch.randn((wk.Nk, wk.Hkv, 128), generator=gen, device=dev).to(torch.bfloat16)
    kc = torch.empty((wk.Hkv, wk.Nk, 128), dtype=torch.int8, device=dev)
    vc = torch.empty_like(kc)
    ks = torch.empty((wk.Hkv, wk.Nk), dtype=torch.float16, device=dev)
    vs = torch.empty_like(ks)
    for _ in range(3):
        qas.int8kv_cache_write(kr, vr, kc, ks, vc, vs, 0, status=status)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(reps):
        qas.int8kv_cache_write(kr, vr, kc, ks, vc, vs, 0, status=status)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / reps
    rows = wk.Nk * wk.Hkv
    nbytes = rows * (2 * 256 + 2 * 128 + 2 * 2)  # bf16 K and V rows in, int8 codes and fp16 scales out
    kv["cache_write_32k_bf16"] = {"ms": ms, "bytes": nbytes, "gbs": nbytes / (ms * 1e-3) / 1e9,
                                  "tokens": wk.Nk, "Hkv": wk.Hkv}
    assert status.item() == 0, "device status set in int8kv_cache_write"

    # ---- per-clock rates of the instructions the dense kernel issues (one CTA per SM)
    probe = {}
    for kind, key, iters in ((0, "f16_mac_per_clk_sm", 50000), (1, "f8_mac_per_clk_sm", 50000),
                             (2, "ex2_per_clk_sm", 1000)):
        qas.sage_probe_rates(kind, max(1, iters // 10), dev)  # warm-up
        r = qas.sage_probe_rates(kind, iters, dev)
        probe[key] = r["per_clock"]
        probe[key.replace("_per_clk_sm", "_probe_mhz")] = r["mhz"]

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    pk = peaks()
    kv["cache_write_32k_bf16"]["frac_hbm"] = kv["cache_write_32k_bf16"]["gbs"] / pk["hbm_gbs"]
    # the preparation against the measured copy bandwidth.  The method's own
    # bytes: Q, K, V read once (bf16), Q/K codes (1 B) and V codes (1 B,
    # padded to 128 tokens) written.  The fused call moves more: K and V are
    # read twice (the mean / amax must be known before any code) and the Q/K
    # codes go out as 2-byte fp16 images, which spares the attention its
    # conversion passes.
    elems = w.B * w.H * w.Nk * 128
    vcodes = w.B * w.H * 128 * qas.nk_pad(w.Nk)
    method_bytes = 3 * elems * 2 + 2 * elems + vcodes
    moved_bytes = 3 * elems * 2 + 2 * elems * 2 + 2 * elems * 2 + vcodes
    ms_p = comp["sage_quantize_qkv_ms"]
    three = comp["three_entry_points"]
    quantizers = {
        "sage_quantize_qkv": {"ms": ms_p, "method_bytes": method_bytes, "moved_bytes": moved_bytes,
                              "gbs_method": method_bytes / (ms_p * 1e-3) / 1e9,
                              "gbs_moved": moved_bytes / (ms_p * 1e-3) / 1e9,
                              "frac_hbm_method": method_bytes / (ms_p * 1e-3) / 1e9 / pk["hbm_gbs"],
                              "frac_hbm_moved": moved_bytes / (ms_p * 1e-3) / 1e9 / pk["hbm_gbs"],
                              "launches": 3},
        "separate": {"sage_quantize_qk_ms": three["sage_quantize_qk_ms"],
                     "sage_quantize_v_ms": three["sage_quantize_v_ms"],
                     "image_passes_ms": three["sage_attn_fwd_ms"] - comp["sage_attn_fwd_f16_ms"],
                     "total_ms": three["step_ms"] - comp["sage_attn_fwd_f16_ms"], "launches": 8}}
    p16 = pk["bf16_tflops"]
    for name in ("prompt32k_q1024", "prompt64k_q512_outliers"):
        # Q.K^T and P.V both on the bf16/f16 tensor path; the fp16 hi/lo split of
        # the P.V weights doubles the P.V MMAs, so the MMA work is 1.5x the formula
        a = kv[name]["tflops_causal"]
        kv[name]["roofline"] = {"bound": "tensor", "achieved": a, "peak": p16, "unit": "TFLOP/s",
                                "frac": a / p16, "mma_frac": 1.5 * a / p16,
                                "peak_note": f"{pk['source']}: bf16 burst; achieved over the causal-visible pairs"}
    # Q.K^T on the f16 tensor path, P.V on FP8 (2x the f16 rate, nominal ratio):
    # equal FLOPs on both, so the effective peak is the harmonic combination.
    peak_mixed = 2.0 / (1.0 / p16 + 1.0 / (2.0 * p16))
    achieved = w.flops / (comp["sage_attn_fwd_f16_ms"] * 1e-3) / 1e12
    sha = kernel_sha("attn_dense.cu")[:16]
    same_src = TRAFFIC["sha256_prefix"] == sha
    traffic = TRAFFIC["bytes"] if same_src else None
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8/fp8 (fp32 accumulate)",
        "data": "synthetic (seeded SplitMix64/Box-Muller, the workload's shapes)",
        "config": {"workload": WORKLOAD, "B": 1, "H": 24, "Nq": 37810, "Nk": 37810, "d": 128, "q_block": 128,
                   "k_block": 128, "causal": False, "l2": "inputs larger than L2 (696 MB of Q/K/V)",
                   "parallelism": (f"heads sharded: {w.H * world} heads over {world} ranks by sage_shard_range, "
                                   "no collective on the data path" if world > 1 else "single GPU")},
        "roofline": {"kernel": "sage_attn_fwd_kernel (tcgen05 attention over the fp16 images, sage_attn_fwd_f16)",
                     "bound": "tensor", "achieved": achieved, "peak": peak_mixed, "unit": "TFLOP/s",
                     "frac": achieved / peak_mixed, "traffic": traffic,
                     "algorithmic_bytes": ATTN_METHOD_BYTES,
                     "traffic_ratio": traffic / ATTN_METHOD_BYTES if traffic else None,
                     "tensor_pipe_active": TRAFFIC["tensor_pipe_active"] if same_src else None,
                     "peak_note": (f"{pk['source']}: bf16 burst {p16} TFLOP/s for the Q.K^T half, x2 (nominal "
                                   f"fp8/bf16 ratio) for the P.V half"),
                     # the softmax's MUFU demand: one ex2 per score
                     "exp2_per_sm_per_clock": (w.B * w.H * w.Nq * w.Nk) / (comp["sage_attn_fwd_f16_ms"] * 1e-3)
                     / (current_sms(dev) * 1e6 * ((clocks or {}).get("sm_mhz") or 2070.0)),
                     # the same call against the tensor core's own rates, measured by the
                     # library's probe (MACs per SM per clock) at the clock sampled in the
                     # timed region
                     "peak_per_clock": probe,
                     "frac_per_clock": achieved / per_clock_peak(probe, current_sms(dev),
                                                                 (clocks or {}).get("sm_mhz") or 2070.0)},
        "components": comp,
        "quantizers": quantizers,
        "causal_lse": causal,
        "int8kv": kv,
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": 4 * args.steps,
    }
    if not args.no_cpu_baseline:
        configs, cb = per_config_results(qas, torch, dev, pk, peak_mixed,
                                         {"dense_out": lambda: qas.sage_attn_fwd(qk, vq, bq, bk, workspace=ws_a),
                                          "attn_ms": attn_each, "step_ms": step_each})
        line["configs"] = configs
        line["cpu_baseline"] = cb
        line["cpu_baseline"]["cpu"] = cpu_model()
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def run_case(args):
    """A small workload for profiler captures: a few calls of one path."""
    import torch

    import quantized_attention_sage_gb300 as qas

    qas.build()
    torch.cuda.set_device(0)
    before = None
    if args.case == "dense":
        w = synth.DenseWorkload("profile_case", 11, 1, args.heads, args.seq, args.seq, 128)
        x = synth.dense_inputs(w)
        q, k, v = (torch.from_numpy(x[t].view(np.int16)).view(torch.bfloat16).cuda() for t in ("q", "k", "v"))
        run = lambda: qas.sage_attention(q, k, v, 128, 128)  # noqa: E731
        flops = w.flops
    elif args.case == "kvcache":
        # int8 KV-cache writer: args.seq tokens x args.heads kv heads of bf16 K and V rows
        gen = torch.Generator(device="cuda")
        gen.manual_seed(5)
        kr = torch.randn((args.seq, args.heads, 128), generator=gen, device="cuda").to(torch.bfloat16)
        vr = torch.randn((args.seq, args.heads, 128), generator=gen, device="cuda").to(torch.bfloat16)
        kc = torch.empty((args.heads, args.seq, 128), dtype=torch.int8, device="cuda")
        vc = torch.empty_like(kc)
        ks = torch.empty((args.heads, args.seq), dtype=torch.float16, device="cuda")
        vs = torch.empty_like(ks)
        flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        before = flush.zero_  # cold L2 for the writer, outside the timed call
        run = lambda: qas.int8kv_cache_write(kr, vr, kc, ks, vc, vs, 0)  # noqa: E731
        flops = 0
    else:
        wk = synth.Int8KVWorkload("profile_case", 12, args.queries, args.seq, args.heads, max(1, args.heads // 4))
        tq, kc, ks, vc, vs = kv_cache_on_device(qas, torch, synth.int8kv_inputs(wk), torch.device("cuda"))
        run = lambda: qas.int8kv_prompt_attn(tq, kc, ks, vc, vs, wk.q_pos0)  # noqa: E731
        flops = wk.flops
    for _ in range(args.reps):
        if before is not None:
            before()
        run()
    torch.cuda.synchronize()
    if before is not None:
        before()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    run()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    res = {"case": args.case, "heads": args.heads, "seq": args.seq, "ms": ms, "tflops": flops / (ms * 1e-3) / 1e12}
    if args.case == "kvcache":
        nbytes = args.seq * args.heads * (2 * 256 + 2 * 128 + 2 * 2)
        res.update(bytes=nbytes, gbs=nbytes / (ms * 1e-3) / 1e9)
    print(json.dumps(res))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--case", choices=["dense", "int8kv", "kvcache"], default=None,
                    help="run a small workload of one path (profiler captures) instead of the bench")
    ap.add_argument("--heads", type=int, default=24)
    ap.add_argument("--seq", type=int, default=8192)
    ap.add_argument("--queries", type=int, default=1024)
    ap.add_argument("--reps", type=int, default=2)
    args = ap.parse_args()
    if args.case:
        run_case(args)
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        run_reference(args, rank)
    else:
        run_ours(args, rank, world)


if __name__ == "__main__":
    main()
