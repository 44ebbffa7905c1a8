#!/usr/bin/env python3
"""Decode-attention layer-step benchmark on GB300.  Prints ONE JSON line.

A step is one pass of the whole hot path over one batch: the paged append of
each sequence's current token (its K/V, or c_KV/k_R, written through the block
table) followed by the decode (split planner, decode kernel, split-KV combine)
over all cached tokens.  Inputs are synthetic, seeded, resident in HBM and far
larger than L2, so every step streams the KV cache from HBM.

  python bench.py [--config llama3_8b] [--steps K] [--warmup W]
  python bench.py --impl reference      # the float64 CPU oracle on a bounded sample
  python bench.py --config llama3_70b --q-len 4   # 4 new tokens per sequence (GQA)
  python bench.py --config deepseek_v3_mla --absorb  # + query absorption, value up-projection
  torchrun --nproc-per-node N bench.py --gpus N   # N independent replicas

Metric: decode-attention KV-read GB/s (algorithmic KV bytes of a step / step
time); also microseconds per layer-step and the fraction of ~8 TB/s.  The
headline times the step captured once in a CUDA graph and replayed, as a
serving loop would run it; the line also carries the same step issued call by
call ("direct").  The roofline times the decode call alone, replayed from a
graph, and the line also gives it with CUDA events around each direct call.

With --q-len L > 1 (GQA only) a step appends the last L tokens of every
sequence and runs the multi-token decode: L queries per sequence, causal among
the new tokens (speculative verification).  The KV bytes read are the same as
for one token; the work per byte is L times larger.

With --absorb (MLA only) a step also runs the per-head projections around
the decode: W_UK^T q^C before it (writing the absorbed query) and W_UV u~
after it, with random bf16 weights of DeepSeek-V3's shapes.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn KV-read GB/s (% of ~8 TB/s HBM) and µs per layer-step"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2**20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="llama3_8b")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--batch", type=int, default=0,
                    help="override the batch size (smaller profiling cases); 0 = the config's")
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=0, help="0 = same as --steps")
    ap.add_argument("--q-len", type=int, default=1,
                    help="new tokens per sequence (GQA; > 1 runs the multi-token decode)")
    ap.add_argument("--prefill", default="",
                    help="B,S,Q: time only the explicit-form MLA prefill of Q new tokens over B "
                         "sequences of S cached rows (DeepSeek-V3 heads) and print its JSON")
    ap.add_argument("--no-all-configs", action="store_true",
                    help="skip timing the decode call of every workload (the all_configs object)")
    ap.add_argument("--absorb", action="store_true",
                    help="MLA: add query absorption and value up-projection to every step")
    return ap.parse_args()


def env_ranks():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def file_hash(*paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def max_over_ranks(x: float, dist, device) -> float:
    """The largest x over all ranks (identity on one process): the slowest
    replica sets the time of the whole job."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_replica: float, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: the bytes every replica read in one step, over the
    step time (already the maximum over ranks)."""
    return bytes_per_replica * world / (ms_per_step * 1e-3) / 1e9


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source(wl) -> str:
    name = "decode_mla.cu" if wl.kind == "mla" else "decode_gqa.cu"
    return os.path.join(ROOT, "kv_cache_decode_paged_gb300", "csrc", name)


def recorded_traffic(wl, config):
    """DRAM bytes per launch of the decode kernel from the committed ncu summary,
    valid only while the kernel source is unchanged since the capture."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f).get(config)
    except Exception:
        return None
    if not rec or rec.get("source_sha") != file_hash(kernel_source(wl)):
        return None
    return rec.get("bytes_per_launch")


class NvmlClocks:
    """SM clock and clock-event reasons read through NVML (libnvidia-ml, read-only
    queries) by a thread that polls every millisecond, so that even a timed
    region of a few milliseconds holds samples."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu_uuid: str):
        import ctypes
        self.samples = []
        self.ok = False
        self._stop = threading.Event()
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            self.dev = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByUUID(gpu_uuid.encode(), ctypes.byref(self.dev)) != 0:
                return
            self.reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint()
            nv.nvmlDeviceGetMaxClockInfo(self.dev, 1, ctypes.byref(mx))   # NVML_CLOCK_SM
            self.max_mhz = float(mx.value)
            self.nv, self.ct = nv, ctypes
            self.ok = True
        except Exception:
            self.ok = False

    def _poll(self):
        ct, nv = self.ct, self.nv
        clk, rs = ct.c_uint(), ct.c_ulonglong()
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(self.dev, 1, ct.byref(clk)) == 0 and \
                    self.reasons_fn(self.dev, ct.byref(rs)) == 0:
                self.samples.append((time.monotonic(), float(clk.value), int(rs.value)))
            time.sleep(0.001)

    def start(self):
        if self.ok:
            threading.Thread(target=self._poll, daemon=True).start()

    def stop(self):
        self._stop.set()

    def summary(self, t0, t1):
        win = [(c, r) for t, c, r in self.samples if t0 <= t <= t1]
        if not win:
            return None
        reasons = sorted({n for _, r in win for bit, n in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(c for c, _ in win), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(win), "window": "timed region",
                "source": "NVML, polled every 1 ms"}


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons in the background,
    with NVML polling beside it for short timed regions."""
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        self.gpu_id = gpu_id
        self.nvml = NvmlClocks(gpu_id)

    def start(self):
        self.nvml.start()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 6:
                self.samples.append((time.monotonic(), parts))

    def stop(self):
        self.nvml.stop()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        fine = self.nvml.summary(t0, t1)
        if fine is not None:
            return fine
        win = [s for t, s in self.samples if t0 <= t <= t1]
        window = "timed region"
        if not win:
            win = [s for _, s in self.samples]
            window = "whole run (no sample fell inside the timed region)"
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "window": "nvidia-smi unavailable"}
        sm = [float(s[0]) for s in win if s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in win if s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in win for i in range(4) if s[2 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(win), "window": window, "source": "nvidia-smi, every 20 ms"}


def config_dict(wl, args):
    d = {"workload": wl.name, "kind": wl.kind, "batch": wl.B, "h": wl.h,
         "block_size": wl.block_size, "kv_dtype": wl.kv_dtype,
         "total_tokens": wl.total_tokens, "kv_bytes_per_step": wl.kv_bytes(),
         "seq_lens": {"min": int(wl.seq_lens.min()), "max": int(wl.seq_lens.max()),
                      "mean": float(wl.seq_lens.mean())},
         "seed": args.seed,
         "l2": (("inputs larger than L2: every step reads %.2f GB of KV vs %d MB of L2"
                 % (wl.kv_bytes() / 1e9, L2_BYTES // 2**20)) if wl.kv_bytes() > L2_BYTES else
                ("inputs smaller than L2 and not flushed: %.1f KB of KV stays L2-resident "
                 "(a launch-bound case, timed for latency)" % (wl.kv_bytes() / 1e3))),
         "parallelism": f"replicas x{args.gpus}"}
    if wl.kind == "gqa":
        d.update({"h_kv": wl.h_kv, "d_h": wl.d})
    if args.q_len > 1:
        d["workload"] = f"{wl.name}, {args.q_len} new tokens per sequence"
        d["q_len"] = args.q_len
    if args.absorb:
        d["workload"] = f"{wl.name}, with query absorption and value up-projection"
        d.update({"d_hc": 128, "d_v": 128, "weights": "random bf16 W_UK [h][128][512], W_UV [h][128][512]"})
    else:
        d.update({"d_c": wl.d_c, "d_rope": wl.d_rope})
    return d


def multi_queries(args, wl):
    """[B][q_len][h][d] bf16 bits for a multi-token run, else None."""
    if args.q_len <= 1:
        return None
    if wl.kind != "gqa":
        raise SystemExit("--q-len > 1 needs a GQA config")
    from kv_cache_decode_paged_gb300 import inputs
    return inputs.multi_token_queries(wl, args.q_len, args.seed)


# ----------------------------------------------------------------------- oracle

def oracle_sample_rate(wl, budget_s, oracle, qm=None):
    """Run the oracle over whole sequences, in a fixed shuffled order and over
    the workload again if it finishes early, until the time budget is spent.
    Returns (GB/s of KV read, seconds, sample description)."""
    done_bytes, t_total, n_seq, passes = 0, 0.0, 0, 0
    per_tok = wl.kv_bytes() / max(1, wl.total_tokens)
    import numpy as np
    order = list(np.random.default_rng(123).permutation(wl.B))
    codes = {}   # E4M3 codes per sequence: the stored cache, made once, untimed
    while t_total < budget_s:
        passes += 1
        for b in order:
            sl = wl.seq_slice(b)
            t0 = time.perf_counter()
            if wl.kind == "mla" and wl.kv_dtype == "fp8":
                if b not in codes:
                    codes[b] = np.concatenate([oracle.quantize_e4m3(wl.c_kv[sl], wl.k_scale),
                                               oracle.quantize_e4m3(wl.k_r[sl], wl.v_scale)], axis=1)
                t0 = time.perf_counter()
                oracle.mla_decode_e4m3(wl.q[b], codes[b], wl.d_c, wl.scale, wl.k_scale, wl.v_scale)
            elif wl.kind == "mla":
                rows = np.concatenate([wl.c_kv[sl], wl.k_r[sl]], axis=1)
                oracle.mla_decode(wl.q[b], rows, wl.d_c, wl.scale)
            elif wl.kv_dtype == "fp8":
                if b not in codes:
                    codes[b] = (oracle.quantize_e4m3(wl.k[sl], wl.k_scale),
                                oracle.quantize_e4m3(wl.v[sl], wl.v_scale))
                kc, vc = codes[b]
                t0 = time.perf_counter()
                if qm is None:
                    oracle.gqa_decode(wl.q[b], kc, vc, wl.scale, fmt=oracle.FMT_E4M3,
                                      k_scale=wl.k_scale, v_scale=wl.v_scale)
                else:
                    oracle.gqa_decode_multi(qm[b], kc, vc, wl.scale, fmt=oracle.FMT_E4M3,
                                            k_scale=wl.k_scale, v_scale=wl.v_scale)
            elif qm is None:
                oracle.gqa_decode(wl.q[b], wl.k[sl], wl.v[sl], wl.scale)
            else:
                oracle.gqa_decode_multi(qm[b], wl.k[sl], wl.v[sl], wl.scale)
            t_total += time.perf_counter() - t0
            done_bytes += int(wl.seq_lens[b]) * per_tok
            n_seq += 1
            if t_total >= budget_s:
                break
    gbs = done_bytes / t_total / 1e9 if t_total > 0 else 0.0
    return gbs, t_total, (f"{n_seq} sequences of the {wl.B} ({passes} pass(es) over the batch, "
                          f"{done_bytes / 1e6:.1f} MB of KV), all heads")


def run_reference(args, wl, rank):
    """The reference arm: the float64 CPU oracle as it stands."""
    import numpy as np
    import oracle
    oracle.build()
    per_tok = wl.kv_bytes() / max(1, wl.total_tokens)
    steps, warm = args.steps, args.warmup
    # size one step (a few KV heads of one sequence) so the whole run ends in ~2 minutes
    budget_per_step = min(0.5, 120.0 / max(1, steps + warm))
    order = list(np.argsort(wl.seq_lens))[len(wl.seq_lens) // 2:] or [0]
    qm = multi_queries(args, wl)
    pj = None
    if args.absorb:
        from kv_cache_decode_paged_gb300 import inputs
        pj = inputs.mla_projections(wl.B, h=wl.h, d_c=wl.d_c, d_rope=wl.d_rope, seed=args.seed)
        f64 = lambda bits: inputs.bf16_to_f32(bits).astype(np.float64)
        w_uk, w_uv = f64(pj.w_uk), f64(pj.w_uv)

    codes = {}

    def fp8_codes(b, heads):
        """The stored E4M3 codes of sequence b's first `heads` KV heads: the
        cache as it sits in memory, made once outside the timed steps (the
        step's own append writes one token per sequence)."""
        if (b, heads) not in codes:
            sl = wl.seq_slice(b)
            codes[(b, heads)] = (oracle.quantize_e4m3(wl.k[sl, :heads], wl.k_scale),
                                 oracle.quantize_e4m3(wl.v[sl, :heads], wl.v_scale))
        return codes[(b, heads)]

    def one(i, heads):
        b = int(order[i % len(order)])
        sl = wl.seq_slice(b)
        if wl.kind == "mla":
            rows = np.concatenate([wl.c_kv[sl], wl.k_r[sl]], axis=1)
            hq = max(1, heads)
            if pj is None and wl.kv_dtype == "fp8":
                if b not in codes:
                    codes[b] = np.concatenate([oracle.quantize_e4m3(wl.c_kv[sl], wl.k_scale),
                                               oracle.quantize_e4m3(wl.k_r[sl], wl.v_scale)], axis=1)
                oracle.mla_decode_e4m3(wl.q[b, :hq], codes[b], wl.d_c, wl.scale, wl.k_scale,
                                       wl.v_scale)
            elif pj is None:
                oracle.mla_decode(wl.q[b, :hq], rows, wl.d_c, wl.scale)
            else:   # absorb, decode, up-project the first hq heads
                qa = np.concatenate([oracle.mla_absorb_query(f64(pj.q_nope[b, :hq]), w_uk[:hq]),
                                     f64(pj.q_rope[b, :hq])], axis=1)
                u, _ = oracle.mla_decode(qa, f64(rows), wl.d_c, wl.scale, fmt=oracle.FMT_F64)
                oracle.mla_apply_wuv(u, w_uv[:hq])
            return int(wl.seq_lens[b]) * per_tok * hq / wl.h
        g = wl.g
        kw = {}
        k, v = wl.k[sl, :heads], wl.v[sl, :heads]
        if wl.kv_dtype == "fp8":
            k, v = fp8_codes(b, heads)
            kw = dict(fmt=oracle.FMT_E4M3, k_scale=wl.k_scale, v_scale=wl.v_scale)
        if qm is None:
            oracle.gqa_decode(wl.q[b, :heads * g], k, v, wl.scale, **kw)
        else:
            oracle.gqa_decode_multi(qm[b, :, :heads * g], k, v, wl.scale, **kw)
        return int(wl.seq_lens[b]) * per_tok * heads / wl.h_kv

    units = wl.h if wl.kind == "mla" else wl.h_kv
    heads = units
    if wl.kv_dtype == "fp8" and wl.kind == "gqa":
        fp8_codes(int(order[0]), heads)
    if wl.kv_dtype == "fp8" and wl.kind == "mla":   # the stored codes, made outside the timed steps
        for i in range(max(warm, steps) + 1):
            b = int(order[i % len(order)])
            if b not in codes:
                sl = wl.seq_slice(b)
                codes[b] = np.concatenate([oracle.quantize_e4m3(wl.c_kv[sl], wl.k_scale),
                                           oracle.quantize_e4m3(wl.k_r[sl], wl.v_scale)], axis=1)
    t0 = time.perf_counter()
    one(0, heads)
    dt = time.perf_counter() - t0
    while heads > 1 and dt * heads / units > budget_per_step and dt > budget_per_step:
        heads = max(1, heads // 2)
        dt /= 2
    if wl.kv_dtype == "fp8" and wl.kind == "gqa":
        codes.clear()
        for i in range(max(warm, steps)):
            fp8_codes(int(order[i % len(order)]), heads)
    for i in range(warm):
        one(i, heads)
    total_bytes = 0.0
    t0 = time.perf_counter()
    for i in range(steps):
        total_bytes += one(i, heads)
    el = time.perf_counter() - t0
    value = total_bytes / el / 1e9
    cores = oracle.num_threads()
    sample = (f"each step: one sequence of the upper half of the length mix, "
              f"{heads} of {units} {'query' if wl.kind == 'mla' else 'KV'} heads")
    line = {"metric": METRIC, "impl": "reference", "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": steps, "warmup": warm,
            "ms_per_step": el / steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(wl, args),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------ every workload

ALL_CONFIGS = ["tiny", "llama3_8b", "llama3_70b", "llama3_70b_fp8", "deepseek_v3_mla",
               "deepseek_v3_mla_fp8", "long_gqa8", "long_mqa"]
# multi-token decode (new tokens verified per pass), timed the same way
MT_CONFIGS = [("llama3_70b", 8), ("llama3_70b_fp8", 8)]
FLUSH_BYTES = 512 * 2**20   # 4x L2


def replay_us(torch, fn, n, stream):
    """Mean microseconds of fn captured once in a CUDA graph and replayed n
    times between two events on `stream`."""
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        fn()
    for _ in range(3):
        gr.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(n):
        gr.replay()
    b.record(stream)
    torch.cuda.synchronize()
    del gr
    return a.elapsed_time(b) / n * 1e3


def time_all_configs(args, sampler, headline, dev):
    """The decode call (planner, decode kernel, combine) of every workload,
    replayed from a CUDA graph: back to back, and after an L2 flush before
    every replay.  The flush reads a buffer 4x the size of L2 (a read leaves
    clean lines behind, so no write-back lands in the decode's time); the
    flush is timed alone the same way and subtracted."""
    import torch

    import kv_cache_decode_paged_gb300 as kv
    from kv_cache_decode_paged_gb300 import inputs
    from kv_cache_decode_paged_gb300.device import GpuWorkload

    peak, _ = hbm_peak()
    stream = torch.cuda.current_stream()
    flush_buf = torch.ones(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    sink = torch.empty((), dtype=torch.int64, device=dev)

    def flush():
        torch.sum(flush_buf, dim=0, dtype=torch.int64, out=sink)

    n = max(50, args.steps)
    res = {}
    for name in ALL_CONFIGS:
        if headline is not None and headline.wl.name == name:
            g = headline
        else:
            g = GpuWorkload(inputs.make_workload(name, seed=args.seed), poison=False, device=dev)
        wl = g.wl
        ws = g.workspace()
        dv = wl.d_c if wl.kind == "mla" else wl.d
        out = torch.empty((wl.B, wl.h, dv), dtype=torch.float32, device=dev)
        lse = torch.empty((wl.B, wl.h), dtype=torch.float32, device=dev)
        desc = g.cache.descriptor()

        def decode():
            if wl.kind == "gqa":
                kv.kvattn_decode_gqa(g.q, desc, g.bt, g.seq_lens, wl.h, wl.h_kv, wl.d, wl.scale,
                                     out, lse, ws, err=g.err)
            else:
                kv.kvattn_decode_mla(g.q, desc, g.bt, g.seq_lens, wl.h, wl.d_c, wl.d_rope,
                                     wl.scale, out, lse, ws, err=g.err)

        def flushed():
            flush()
            decode()

        torch.cuda.synchronize()
        t0 = time.monotonic()
        warm = replay_us(torch, decode, n, stream)
        both = replay_us(torch, flushed, n, stream)
        alone = replay_us(torch, flush, n, stream)
        t1 = time.monotonic()
        cold = max(both - alone, 1e-3)
        kvb = wl.kv_bytes()
        target = 0.65 if wl.kind == "mla" else 0.75
        fp8 = wl.kv_dtype == "fp8"
        entry = {"kernel": ("MLA absorbed decode" if wl.kind == "mla" else "GQA decode") +
                           (", FP8-E4M3 cache" if fp8 else ""),
                 "batch": wl.B, "h": wl.h, "kv_bytes": kvb, "total_tokens": wl.total_tokens,
                 "us_decode_call": cold, "us_decode_call_back_to_back": warm,
                 "us_l2_flush": alone,
                 "gbs": kvb / cold / 1e3, "frac_of_measured_hbm": kvb / cold / 1e3 / peak,
                 "pct_of_8tbs": 100.0 * kvb / cold / 1e3 / NOMINAL_HBM_GBS,
                 "gbs_back_to_back": kvb / warm / 1e3, "target_frac": target,
                 "traffic": recorded_traffic(wl, name),
                 "clocks": sampler.summary(t0, t1), "device_err_bits": g.err_bits()}
        if wl.kind == "gqa":
            entry["h_kv"] = wl.h_kv
        if name == "tiny":
            entry["note"] = "launch-bound: 70 KB of KV, timed for latency"
        res[name] = entry
        del out, lse, ws, decode, flushed
        if g is not headline:
            del g
        torch.cuda.empty_cache()
    for name, q_len in MT_CONFIGS:
        res[f"{name}_q{q_len}"] = time_multi_token(name, q_len, args, sampler, dev, stream, peak,
                                                   flush, n)
        torch.cuda.empty_cache()
    res["mla_prefill"] = time_prefill(args, sampler, dev, stream, flushed_by=(flush, n))
    res["how"] = ("decode call replayed from a CUDA graph %d times; us_decode_call = (flush + "
                  "decode replays - flush replays) / %d with an L2 flush (sum over a %d MB "
                  "buffer) before every decode; gbs, frac and pct use it" % (n, n,
                                                                             FLUSH_BYTES >> 20))
    return res


def time_multi_token(name, q_len, args, sampler, dev, stream, peak, flush, n):
    """The multi-token decode call of a GQA workload (q_len new tokens per
    sequence, the last q_len cached ones), back to back and after an L2 flush,
    as for the single-token entries."""
    import torch

    import kv_cache_decode_paged_gb300 as kv
    from kv_cache_decode_paged_gb300 import inputs
    from kv_cache_decode_paged_gb300.device import GpuWorkload, dev_bits

    wl = inputs.make_workload(name, seed=args.seed)
    g = GpuWorkload(wl, poison=False, device=dev)
    qm = dev_bits(inputs.multi_token_queries(wl, q_len, args.seed), dev)
    ws = kv.workspace_for(kv.KVATTN_GQA, wl.B, wl.h * q_len, wl.h_kv, wl.d, 0, dev)
    out = torch.empty((wl.B, q_len, wl.h, wl.d), dtype=torch.float32, device=dev)
    lse = torch.empty((wl.B, q_len, wl.h), dtype=torch.float32, device=dev)
    desc = g.cache.descriptor()

    def decode():
        kv.kvattn_decode_gqa_multi(qm, desc, g.bt, g.seq_lens, q_len, wl.h, wl.h_kv, wl.d,
                                   wl.scale, out, lse, ws, err=g.err)

    def flushed():
        flush()
        decode()

    torch.cuda.synchronize()
    t0 = time.monotonic()
    warm = replay_us(torch, decode, n, stream)
    both = replay_us(torch, flushed, n, stream)
    alone = replay_us(torch, flush, n, stream)
    t1 = time.monotonic()
    cold = max(both - alone, 1e-3)
    kvb = wl.kv_bytes()
    rows = q_len * wl.h // wl.h_kv
    fp8 = wl.kv_dtype == "fp8"
    return {"kernel": "GQA multi-token decode" + (", FP8-E4M3 cache" if fp8 else "") +
                      (" (tcgen05)" if rows > (16 if fp8 else 32) else " (mma.sync)"),
            "batch": wl.B, "h": wl.h, "h_kv": wl.h_kv, "q_len": q_len, "rows_per_unit": rows,
            "kv_bytes": kvb, "us_decode_call": cold, "us_decode_call_back_to_back": warm,
            "us_l2_flush": alone, "gbs": kvb / cold / 1e3,
            "frac_of_measured_hbm": kvb / cold / 1e3 / peak,
            "pct_of_8tbs": 100.0 * kvb / cold / 1e3 / NOMINAL_HBM_GBS,
            "gbs_back_to_back": kvb / warm / 1e3,
            "flop_per_byte": 4.0 * wl.d * rows / (2.0 * wl.d * (1 if fp8 else 2)),
            "clocks": sampler.summary(t0, t1), "device_err_bits": g.err_bits()}


def prefill_flops(S, q_len, h, B):
    """FLOPs of one explicit-form MLA prefill call as the kernel performs them:
    the expansion of every 128-row tile of keys and values each (128 new
    tokens, head) visits (2 * 128 * 128 * 512 * 2 per tile), plus the causal
    attention proper (2 * (192 + 128) per visible (token, row) pair), over all
    heads and sequences."""
    tiles = sum((S - q_len + min(q_len, 128 * qt + 128) + 127) // 128
                for qt in range((q_len + 127) // 128))
    expand = tiles * 128 * 128 * 512 * 2 * 2 * h * B
    attend = sum(S - q_len + j + 1 for j in range(q_len)) * (192 + 128) * 2 * h * B
    return expand, attend


def time_prefill(args, sampler, dev, stream, flushed_by=None, B=4, S=4096, q_len=512):
    """Explicit-form MLA prefill at DeepSeek-V3 shapes: B sequences of S cached
    rows (the last q_len of them new), 128 heads, replayed from a CUDA graph
    after an L2 flush like the decode calls."""
    import torch

    import kv_cache_decode_paged_gb300 as kv
    from kv_cache_decode_paged_gb300 import inputs
    from kv_cache_decode_paged_gb300.device import GpuWorkload, dev_bits

    if flushed_by is None:
        flush_buf = torch.ones(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
        sink = torch.empty((), dtype=torch.int64, device=dev)

        def flush():
            torch.sum(flush_buf, dim=0, dtype=torch.int64, out=sink)
        n = max(50, args.steps)
    else:
        flush, n = flushed_by
    wl = inputs.make_workload("deepseek_v3_mla", seed=args.seed, lens=[S] * B)
    g = GpuWorkload(wl, poison=False, device=dev)
    h = 128
    qn, qr = inputs.prefill_queries(B, q_len, h=h, seed=args.seed)
    pj = inputs.mla_projections(1, h=h, seed=args.seed)
    qn, qr = dev_bits(qn, dev), dev_bits(qr, dev)
    wk, wv = dev_bits(pj.w_uk, dev), dev_bits(pj.w_uv, dev)
    out = torch.empty((B, q_len, h, 128), dtype=torch.float32, device=dev)
    lse = torch.empty((B, q_len, h), dtype=torch.float32, device=dev)
    desc = g.cache.descriptor()

    def run():
        kv.kvattn_mla_prefill(qn, qr, desc, g.bt, g.seq_lens, wk, wv, wl.scale, out, lse,
                              err=g.err)

    def flushed():
        flush()
        run()

    torch.cuda.synchronize()
    t0 = time.monotonic()
    reps = max(10, n // 5)
    warm = replay_us(torch, run, reps, stream)
    both = replay_us(torch, flushed, reps, stream)
    alone = replay_us(torch, flush, reps, stream)
    t1 = time.monotonic()
    cold = max(both - alone, 1e-3)
    expand, attend = prefill_flops(S, q_len, h, B)
    peak = 1928.9
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak = float(json.load(f)["bf16_tflops"])
    except Exception:
        pass
    tf = (expand + attend) / cold / 1e6
    return {"kernel": "explicit-form MLA prefill (keys and values expanded per tile on the SM)",
            "batch": B, "cached_rows": S, "q_len": q_len, "h": h, "us": cold,
            "us_back_to_back": warm, "flop_expand": expand, "flop_attention": attend,
            "tflops": tf, "roofline": {"bound": "tensor", "achieved": tf, "peak": peak,
                                       "unit": "TFLOP/s", "frac": tf / peak,
                                       "peak_source": "MEASURED_PEAKS.json bf16_tflops (burst)"},
            "clocks": sampler.summary(t0, t1), "device_err_bits": g.err_bits()}


# -------------------------------------------------------------------------- ours

def run_ours(args, wl, rank, world, local):
    import numpy as np
    import torch

    import kv_cache_decode_paged_gb300 as kv
    from kv_cache_decode_paged_gb300 import inputs
    from kv_cache_decode_paged_gb300.device import GpuWorkload, dev_bits

    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(dev))

    kv.load_library()
    g = GpuWorkload(wl, poison=False, device=dev)     # pools filled by kvattn_append (untimed)
    torch.cuda.synchronize()

    # the new tokens of every non-empty sequence: positions s_b - L .. s_b - 1
    # (L = 1 for plain decode; clipped at 0 for sequences shorter than L)
    L = args.q_len
    qm = multi_queries(args, wl)
    idx = [(b, t) for b in np.nonzero(wl.seq_lens > 0)[0]
           for t in range(max(0, int(wl.seq_lens[b]) - L), int(wl.seq_lens[b]))]
    live = np.array([b for b, _ in idx], dtype=np.int64)
    tpos = np.array([t for _, t in idx], dtype=np.int64)
    last = wl.cu_seqlens[live] + tpos
    seq_idx = torch.from_numpy(live.astype(np.int32)).to(dev)
    pos = torch.from_numpy(tpos.astype(np.int32)).to(dev)
    if wl.kind == "gqa":
        new0, new1 = dev_bits(wl.k[last], dev), dev_bits(wl.v[last], dev)
        dv = wl.d
    else:
        new0, new1 = dev_bits(wl.c_kv[last], dev), dev_bits(wl.k_r[last], dev)
        dv = wl.d_c
    if qm is None:
        ws = g.workspace()
        out = torch.empty((wl.B, wl.h, dv), dtype=torch.float32, device=dev)
        lse = torch.empty((wl.B, wl.h), dtype=torch.float32, device=dev)
        q_dev = g.q
    else:
        ws = kv.workspace_for(kv.KVATTN_GQA, wl.B, wl.h * L, wl.h_kv, wl.d, 0, dev)
        out = torch.empty((wl.B, L, wl.h, dv), dtype=torch.float32, device=dev)
        lse = torch.empty((wl.B, L, wl.h), dtype=torch.float32, device=dev)
        q_dev = dev_bits(qm, dev)
    desc = g.cache.descriptor()
    # Every call below enqueues on the current stream: this one, or the capture
    # stream while the step is captured in a CUDA graph.
    stream = torch.cuda.current_stream()
    launches = 4 if wl.kind == "gqa" else 3   # append, planner, decode (, combine)
    proj = None
    if args.absorb:
        if wl.kind != "mla":
            raise SystemExit("--absorb needs an MLA config")
        pj = inputs.mla_projections(wl.B, h=wl.h, d_c=wl.d_c, d_rope=wl.d_rope, seed=args.seed)
        proj = {"q_nope": dev_bits(pj.q_nope, dev), "q_rope": dev_bits(pj.q_rope, dev),
                "w_uk": dev_bits(pj.w_uk, dev), "w_uv": dev_bits(pj.w_uv, dev),
                "v": torch.empty((wl.B, wl.h, pj.w_uv.shape[1]), dtype=torch.float32, device=dev)}
        launches += 2
        pev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
                torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]

    def decode():
        if qm is not None:
            kv.kvattn_decode_gqa_multi(q_dev, desc, g.bt, g.seq_lens, L, wl.h, wl.h_kv, wl.d,
                                       wl.scale, out, lse, ws, err=g.err)
        elif wl.kind == "gqa":
            kv.kvattn_decode_gqa(g.q, desc, g.bt, g.seq_lens, wl.h, wl.h_kv, wl.d, wl.scale,
                                 out, lse, ws, err=g.err)
        else:
            kv.kvattn_decode_mla(g.q, desc, g.bt, g.seq_lens, wl.h, wl.d_c, wl.d_rope, wl.scale,
                                 out, lse, ws, err=g.err)

    def step(ev=None, pe=None):
        if proj is not None:
            if pe is not None:
                pe[0].record(stream)
            kv.kvattn_mla_absorb_q(proj["q_nope"], proj["q_rope"], proj["w_uk"], g.q, err=g.err)
            if pe is not None:
                pe[1].record(stream)
        kv.kvattn_append(desc, new0, new1, seq_idx, pos, g.bt, err=g.err)
        if ev is not None:
            ev[0].record(stream)
        decode()
        if ev is not None:
            ev[1].record(stream)
        if proj is not None:
            if pe is not None:
                pe[2].record(stream)
            kv.kvattn_mla_up_v(out, proj["w_uv"], proj["v"], err=g.err)
            if pe is not None:
                pe[3].record(stream)

    gpu_id = "GPU-" + str(torch.cuda.get_device_properties(local).uuid).replace("GPU-", "")
    sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.3)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    w0 = time.monotonic()
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i], pev[i] if proj is not None else None)
    t_end.record(stream)
    torch.cuda.synchronize()
    w1 = time.monotonic()
    if dist:
        dist.barrier()
    ms_total = max_over_ranks(t_start.elapsed_time(t_end), dist, dev)
    dec_ms = [a.elapsed_time(b) for a, b in evs]

    # ---- the headline: the same step captured once in a CUDA graph and
    # replayed, as a serving loop runs it (every kernel of the step still runs
    # on every replay; only the host's per-launch cost between them is gone)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(max(3, args.warmup)):
        graph.replay()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wg0 = time.monotonic()
    g0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    wg1 = time.monotonic()
    if dist:
        dist.barrier()
    graph_ms = max_over_ranks(g0.elapsed_time(g1) / args.steps, dist, dev)
    del graph

    # ---- the decode call alone (planner, decode kernel, combine), replayed
    # from a graph: its duration without the launch gap that events placed
    # around each direct call also count; this times the roofline
    dgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(dgraph):
        decode()
    for _ in range(3):
        dgraph.replay()
    torch.cuda.synchronize()
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    d0.record(stream)
    for _ in range(args.steps):
        dgraph.replay()
    d1.record(stream)
    torch.cuda.synchronize()
    dec_graph_ms = d0.elapsed_time(d1) / args.steps
    del dgraph
    time.sleep(0.05)
    clocks = sampler.summary(wg0, wg1)
    clocks_direct = sampler.summary(w0, w1)
    err_bits = g.err_bits()

    # ---- end to end: host buffers in, result out, every step
    e2e_steps = args.e2e_steps or args.steps
    # (device tensor, pinned host copy) of every input a step reads and every
    # result it returns
    if proj is None:
        dev_in = [q_dev]
        dev_out = [out, lse]
    else:   # the absorbed query is made on the device from q^C and q^R
        dev_in = [proj["q_nope"], proj["q_rope"]]
        dev_out = [proj["v"], lse]
    dev_in += [new0, new1, pos, g.seq_lens]
    h_in = [t.cpu().pin_memory() for t in dev_in]
    h_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in dev_out]
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = sum(t.numel() * t.element_size() for t in h_out)

    def e2e_step():
        for d, hst in zip(dev_in, h_in):
            d.copy_(hst, non_blocking=True)
        step()
        for hst, d in zip(h_out, dev_out):
            hst.copy_(d, non_blocking=True)

    for _ in range(max(3, args.warmup // 4)):
        e2e_step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dist, dev)
    if dist:
        dist.barrier()

    if rank != 0:
        sampler.stop()
        if dist:
            dist.destroy_process_group()
        return

    kvb = wl.kv_bytes()
    ms_direct = ms_total / args.steps
    ms_step = graph_ms
    value = whole_job_gbs(kvb, world, ms_step)
    dec_mean = statistics.mean(dec_ms)
    achieved = kvb / (dec_graph_ms * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if wl.kv_dtype == "bf16" else "fp8-e4m3 cache, bf16 q",
        "data": "synthetic", "config": config_dict(wl, args),
        "us_per_layer_step": ms_step * 1e3,
        "us_decode_call": dec_graph_ms * 1e3,
        "us_decode_call_direct": dec_mean * 1e3,
        "pct_of_8tbs": 100.0 * (value / world) / NOMINAL_HBM_GBS,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "traffic": recorded_traffic(wl, args.config),
                     "kernel": ("decode call (planner + decode kernel + combine) replayed from a "
                                "CUDA graph, CUDA events over --steps replays"),
                     "algorithmic_bytes_per_launch": kvb},
        "e2e": {"value": whole_job_gbs(kvb, world, e2e_ms), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms},
        "timing": ("the step (append + decode call) captured once in a CUDA graph and "
                   "replayed --steps times; 'direct' is the same step issued call by call; "
                   "us_decode_call_direct has CUDA events around each direct decode call"),
        "direct": {"us_per_layer_step": ms_direct * 1e3,
                   "value": whole_job_gbs(kvb, world, ms_direct), "unit": "GB/s",
                   "clocks": clocks_direct},
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
        "device_err_bits": err_bits,
    }
    if proj is not None:
        a_us = statistics.mean(a.elapsed_time(b) for a, b, _, _ in pev) * 1e3
        u_us = statistics.mean(c.elapsed_time(d) for _, _, c, d in pev) * 1e3
        B, h = wl.B, wl.h
        a_bytes = 2 * (h * 128 * wl.d_c + B * h * 128 + B * h * wl.d_rope + B * h * wl.d)
        u_bytes = 2 * h * 128 * wl.d_c + 4 * B * h * wl.d_c + 4 * B * h * 128
        flops = 2 * B * h * 128 * wl.d_c
        line["projections"] = {
            "absorb_q": {"us": a_us, "bytes": a_bytes, "gbs": a_bytes / a_us / 1e3,
                         "frac_of_hbm": a_bytes / a_us / 1e3 / peak, "tflops": flops / a_us / 1e6},
            "up_v": {"us": u_us, "bytes": u_bytes, "gbs": u_bytes / u_us / 1e3,
                     "frac_of_hbm": u_bytes / u_us / 1e3 / peak, "tflops": flops / u_us / 1e6},
            "note": "CUDA events around each launch; bytes = weights + activations read and written"}
    if world == 1 and not args.no_all_configs and args.q_len == 1 and not args.absorb:
        line["all_configs"] = time_all_configs(args, sampler, g, dev)
    sampler.stop()
    if world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        gbs, secs, sample = oracle_sample_rate(wl, args.cpu_budget_s, oracle, qm)
        line["cpu_baseline"] = {"value": gbs, "unit": "GB/s", "cores": oracle.num_threads(),
                                "kind": "oracle", "sample": sample, "seconds": secs}
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def run_prefill_only(args):
    import torch
    torch.cuda.set_device(0)
    import kv_cache_decode_paged_gb300 as kv
    kv.load_library()
    B, S, Q = (int(x) for x in args.prefill.split(","))
    gpu_id = "GPU-" + str(torch.cuda.get_device_properties(0).uuid).replace("GPU-", "")
    sampler = ClockSampler(gpu_id)
    sampler.start()
    res = time_prefill(args, sampler, "cuda:0", torch.cuda.current_stream(), B=B, S=S, q_len=Q)
    sampler.stop()
    print(json.dumps({"metric": "explicit-form MLA prefill TFLOP/s", "value": res["tflops"],
                      "unit": "TFLOP/s", "n_gpus": 1, "higher_is_better": True,
                      "dtype": "bf16", "data": "synthetic", "prefill": res}), flush=True)


def main():
    args = parse()
    rank, world, local = env_ranks()
    if args.prefill and args.impl == "ours":
        if rank == 0:
            run_prefill_only(args)
        return
    from kv_cache_decode_paged_gb300 import inputs
    batch = args.batch or None
    if args.impl == "reference":
        if rank != 0:
            return
        wl = inputs.make_workload(args.config, seed=args.seed, batch=batch)
        run_reference(args, wl, rank)
        return
    wl = inputs.make_workload(args.config, seed=args.seed, batch=batch)
    run_ours(args, wl, rank, world, local)


if __name__ == "__main__":
    main()
