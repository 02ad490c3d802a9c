"""Benchmark of the GB300 TurboQuant KV codec: encode + decode throughput.

One step = encode then decode of the whole long-context serving cache: K, V
[32, 8, 8192, 128] bf16 (N(0, 0.5^2)) into a packed cache of capacity
8192 + 64 tokens, keys 8-bit signed, values 8-bit, then the decode of the
8192 tokens back to bf16 (one launch each; 1.66 GB of algorithmic traffic per
launch, far above the L2). The metric is tokens per second: one token = one
(sequence, position), all 8 KV heads, K and V, encoded and decoded.

Output: one JSON line (rank 0). Fields beyond the metric:
  roofline      the dominant kernel's algorithmic bytes per launch over its
                average launch time (CUDA events on its stream, inside the
                timed region), against the measured HBM copy bandwidth
                (MEASURED_PEAKS.json);
  e2e           the same metric through the Python API with pinned host
                buffers: host->device copy of K, V and device->host copy of
                the decoded K, V inside the timed region;
  cpu_baseline  the oracle (single-threaded C) on a bounded sample of the
                same workload, on this machine's host cores;
  secondary     the other configurations, each with its own roofline: the
                long-context cache at 3-bit values, the Llama-3-8B-shaped
                layer (32 layers per step in CUDA graphs), head_dim 256 and
                512, decode-step appends, fused decode attention, the
                continuous-batching merge and the Lloyd-Max fit;
  clocks        nvidia-smi samples taken during the timed region.
``--impl reference`` times the oracle alone as the reference arm, on the
same configuration. Multi-GPU (torchrun): every rank runs an independent
replica of the workload (weak scaling; the codec has no cross-row exchange),
timed between barriers, max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE = "long_context"  # the largest single-GPU configuration
HEADLINE_V_BITS = 8
LAYERS = 32  # Llama-3-8B-shaped model: layers per secondary step
METRIC = "TurboQuant KV encode/decode tokens/s; achieved HBM GB/s vs GB300 peak"
FALLBACK_HBM_GBS = 6800.0
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
E2E_CHUNK = 4  # sequences per pipelined chunk of the end-to-end step


def r4(x):
    """x to four significant digits (keeps the JSON line short)."""
    return None if x is None else float("%.4g" % x)


def headline_config():
    """The configuration both arms report (identical dicts)."""
    from turboquant_kv_cache_tq_gb300.workloads import WORKLOADS

    w = WORKLOADS[HEADLINE]
    return {"workload": HEADLINE, "shape": [w.B, w.H, w.T, w.D], "t_cap": w.t_cap, "k_bits": w.k_bits,
            "k_signed": w.k_signed, "v_bits": HEADLINE_V_BITS, "in_dtype": "bf16", "out_dtype": "bf16",
            "step": "encode of the whole cache, then its decode (one launch each)",
            "l2": "inputs larger than L2: 1.07 GB of K, V in and out per launch"}


# ---- multi-rank plumbing (host logic; tested with gloo on CPU) --------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), ws, int(os.environ.get("LOCAL_RANK", "0"))


def init_dist(backend: str):
    rank, ws, _ = dist_env()
    if ws > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)
    return rank, ws


def barrier():
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.barrier()


def max_over_ranks(x: float, device="cpu") -> float:
    """The largest value of x over all ranks (x itself without a process group)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, device="cpu") -> float:
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


# ---- byte accounting ------------------------------------------------------------
def bytes_per_row(D: int, k_bits: int, v_bits: int, io_bytes: int) -> int:
    """Algorithmic HBM bytes of one (b,h,t) row for encode (and for decode):
    K and V rows in (out), packed K and V codes, fp16 K scale + zero and V scale."""
    G = D // 32
    return 2 * D * io_bytes + D * k_bits // 8 + D * v_bits // 8 + 2 * G * 2 + G * 2


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def _code_only(text: str) -> str:
    """C++/CUDA source without its comments and with whitespace runs collapsed:
    what the compiler sees, so that a comment edit does not count as a kernel
    change. String literals are kept as they are."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"':
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash() -> str:
    """Hash of the kernel sources (every file of the package's csrc folder,
    comments and layout left out)."""
    csrc = os.path.join(ROOT, "turboquant_kv_cache_tq_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(key: str):
    """dram bytes per launch ("<kernel>@<workload>") from a committed ncu
    summary, if it was taken on the current kernel sources; else None."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(key)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


# ---- clocks -----------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.seek(0)
        rows = [r.split(", ") for r in self.file.read().strip().splitlines() if r.count(",") >= 8]
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows]
        mx = [float(r[2]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        loaded = [s for s, r in zip(sm, rows) if float(r[3]) > 200.0] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx), "reasons": reasons,
                "samples": len(rows)}


# ---- CPU baseline (the oracle) ------------------------------------------------------
def oracle_timing(rows_target: int, min_seconds: float, max_seconds: float, workload: str = HEADLINE,
                  v_bits: int = HEADLINE_V_BITS):
    """Time the oracle's encode + decode on row chunks of the workload until
    min_seconds have passed; returns (rows, seconds)."""
    import oracle
    from turboquant_kv_cache_tq_gb300.workloads import WORKLOADS, make_kv, to_oracle

    w = WORKLOADS[workload]
    chunk_T = 256
    k, v = make_kv(w, B=1, T=chunk_T)  # [1, H, 256, D]: 2048 rows per chunk at H = 8
    ko, vo = to_oracle(k), to_oracle(v)
    oracle.lib()
    done, t0 = 0, time.perf_counter()
    while True:
        cache = oracle.encode_kv(ko, vo, w.k_bits, w.k_signed, v_bits)
        oracle.decode_kv(cache, chunk_T, w.k_bits, w.k_signed, v_bits, out_dtype=oracle.BF16)
        done += ko.shape[1] * chunk_T
        el = time.perf_counter() - t0
        if (el >= min_seconds and done >= min(rows_target, 2048)) or el >= max_seconds:
            return done, el


def _oracle_worker(seconds: float):
    return oracle_timing(2048, seconds, 3 * seconds)


def oracle_all_cores(seconds: float):
    """The same oracle, one process per host core (spawned: no GPU state is
    inherited), each timing its own chunks; rows/s summed. A timing baseline
    only: parity uses the single-threaded oracle."""
    import multiprocessing as mp

    n = os.cpu_count() or 1
    with mp.get_context("spawn").Pool(n) as pool:
        res = pool.map(_oracle_worker, [seconds] * n)
    return sum(r / s for r, s in res), n


def cpu_baseline_obj(rows_per_s: float, H: int, sample: str, all_cores=None):
    d = {"value": r4(rows_per_s / H), "unit": "tokens/s", "cores": 1, "host_cores": os.cpu_count(),
         "kind": "oracle", "sample": sample}
    if all_cores is not None:
        d["all_cores"] = {"value": r4(all_cores[0] / H), "cores": all_cores[1],
                          "note": "one oracle process per host core, rows/s summed"}
    return d


def run_reference(args):
    """The reference arm: the oracle, timed as it stands on the host cores,
    on the headline configuration."""
    rank, ws, _ = dist_env()
    if rank != 0:
        return
    from turboquant_kv_cache_tq_gb300.workloads import WORKLOADS

    w = WORKLOADS[HEADLINE]
    per_step_budget = max(0.02, 150.0 / max(1, args.steps + args.warmup))
    # calibrate: rows the oracle encodes + decodes per second
    rows, secs = oracle_timing(2048, 0.5, 5.0)
    rate = rows / secs
    step_rows = max(2048, int(rate * per_step_budget) // 2048 * 2048)
    for _ in range(args.warmup):
        oracle_timing(step_rows, 0.0, per_step_budget * 2)
    total_rows, total_s = 0, 0.0
    for _ in range(args.steps):
        r, s = oracle_timing(step_rows, per_step_budget, per_step_budget * 4)
        total_rows += r
        total_s += s
    value = total_rows / w.H / total_s
    per_step = total_rows // max(1, args.steps)
    sample = ("%d rows (%d tokens) of %s per step on average, encode+decode at %d-bit values, bf16 out, "
              "single-threaded; tokens/s of that sample" % (per_step, per_step // w.H, HEADLINE, HEADLINE_V_BITS))
    cpu = cpu_baseline_obj(total_rows / total_s, w.H, sample)
    line = {
        "impl": "reference", "metric": METRIC, "value": r4(value), "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": r4(1e3 * total_s / max(1, args.steps)),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": headline_config(), "cpu_baseline": cpu,
        "e2e": {"value": r4(value), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---- the GPU arm --------------------------------------------------------------------
def roofline_obj(kernel: str, workload: str, bytes_per_launch: int, launch_us: float, peak: float, peak_kind: str):
    achieved = bytes_per_launch / (launch_us * 1e-6) / 1e9
    return {"bound": "hbm", "achieved": r4(achieved), "peak": peak, "unit": "GB/s", "frac": r4(achieved / peak),
            "traffic": profiled_traffic("%s@%s" % (kernel, workload)), "kernel": kernel, "peak_source": peak_kind,
            "bytes_per_launch": bytes_per_launch, "launch_us": r4(launch_us)}


def codec_roofline(workload: str, vb: int, rows: int, D: int, kb: int, enc_us: float, dec_us: float, peak,
                   peak_kind):
    """Roofline object of the slower of a workload's encode and decode
    launches, plus both launch times."""
    bpl = rows * bytes_per_row(D, kb, vb, 2)
    name = "%s_v%d" % (workload, vb)
    # the benchmark workloads' decodes (bf16 outputs, whole aligned tiles) take the bulk-copy kernel
    kernel, us = ("encode_kernel", enc_us) if enc_us >= dec_us else ("decode_bulk_kernel", dec_us)
    r = roofline_obj(kernel, name, bpl, us, peak, peak_kind)
    r["encode_us"], r["decode_us"] = r4(enc_us), r4(dec_us)
    r["encode_frac"] = r4(bpl / (enc_us * 1e-6) / 1e9 / peak)
    r["decode_frac"] = r4(bpl / (dec_us * 1e-6) / 1e9 / peak)
    return r


def run_ours(args):
    import turboquant_kv_cache_tq_gb300 as tq
    from turboquant_kv_cache_tq_gb300 import build as tq_build
    from turboquant_kv_cache_tq_gb300.workloads import WORKLOADS, make_kv

    rank, ws, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    rank, ws = init_dist("nccl")
    dev = torch.device("cuda", local)
    if rank == 0 or not os.path.exists(tq.LIB_PATH):
        tq_build.build()
    barrier()
    tq.lib()
    peak, peak_kind = measured_hbm_peak()

    w = WORKLOADS[HEADLINE]
    kb, ks, vb = w.k_bits, w.k_signed, HEADLINE_V_BITS
    B, H, T, D, t_cap = w.B, w.H, w.T, w.D, w.t_cap
    k, v = make_kv(w, device=dev, seed=w.seed + 1000 * rank)
    cache = tq.alloc_cache(B, H, t_cap, D, kb, vb, device=dev)
    ko, vo = torch.empty_like(k), torch.empty_like(v)
    stream = torch.cuda.Stream(device=dev)

    def enc():
        tq.tq_encode_kv(k, v, kb, ks, vb, cache, stream=stream)

    def dec():
        tq.tq_decode_kv(cache, T, kb, ks, vb, out_dtype=torch.bfloat16, k_out=ko, v_out=vo, stream=stream)

    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            enc()
            dec()
    torch.cuda.synchronize(dev)

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        barrier()
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            for e in ev:
                e[0].record(stream)
                enc()
                e[1].record(stream)
                dec()
                e[2].record(stream)
        torch.cuda.synchronize(dev)
        barrier()
    enc_us = 1e3 * sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps
    dec_us = 1e3 * sum(e[1].elapsed_time(e[2]) for e in ev) / args.steps
    total_ms = max_over_ranks(ev[0][0].elapsed_time(ev[-1][2]), dev)
    clocks = clk.summary()
    value = B * T * args.steps * ws / (total_ms / 1e3)
    roofline = codec_roofline(HEADLINE, vb, w.rows, D, kb, enc_us, dec_us, peak, peak_kind)

    # ---- e2e through the Python API with pinned host buffers
    units = [dict(k=k[b:b + E2E_CHUNK], v=v[b:b + E2E_CHUNK], ko=ko[b:b + E2E_CHUNK], vo=vo[b:b + E2E_CHUNK],
                  cache={n: t[b:b + E2E_CHUNK] for n, t in cache.items()}) for b in range(0, B, E2E_CHUNK)]
    e2e = run_e2e(args, tq, units, kb, ks, vb, T, dev, stream)
    e2e_ms = max_over_ranks(e2e["ms"], dev)
    e2e_value = B * T * e2e["steps"] * ws / (e2e_ms / 1e3)
    del units, k, v, ko, vo, cache
    torch.cuda.empty_cache()

    secondary = run_secondary(args, tq, dev, stream, peak, peak_kind, rank) if args.workloads else None

    cpu = None
    if rank == 0 and ws == 1:
        rows_done, secs = oracle_timing(w.rows, args.cpu_seconds, 3 * args.cpu_seconds)
        allc = oracle_all_cores(min(args.cpu_seconds, 5.0)) if args.cpu_all_cores else None
        cpu = cpu_baseline_obj(rows_done / secs, H,
                               "%d rows (%d tokens) of %s, encode+decode at %d-bit values, bf16 out, "
                               "single-threaded; tokens/s of that sample" % (rows_done, rows_done // H, HEADLINE, vb),
                               allc)

    if rank == 0:
        line = {
            "metric": METRIC, "value": r4(value), "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": r4(total_ms / args.steps), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": headline_config(),
            "roofline": roofline,
            "e2e": {"value": r4(e2e_value), "unit": "tokens/s", "h2d_bytes_per_step": e2e["h2d"],
                    "d2h_bytes_per_step": e2e["d2h"]},
            "cpu_baseline": cpu,
            "gpu_launches": 2 * args.steps,
            "clocks": clocks,
            "secondary": secondary,
        }
        print(json.dumps(line, separators=(",", ":")), flush=True)
    barrier()
    if torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


def _time_launches(fn, stream, reps):
    """Average ms of fn() (one launch) over reps back-to-back launches, events on `stream`."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        fn()
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / reps


def run_secondary(args, tq, dev, stream, peak, peak_kind, rank):
    """The other configurations, each with its own roofline object."""
    from turboquant_kv_cache_tq_gb300.workloads import WORKLOADS, make_append_steps, make_kv

    out = {}
    out["llama3_8b_layer_v3"] = time_layers(tq, dev, stream, peak, peak_kind, rank)
    for name in ("long_context", "hd256", "hd512"):
        w = WORKLOADS[name]
        k, v = make_kv(w, device=dev)
        ko, vo = torch.empty_like(k), torch.empty_like(v)
        t_cap = w.t_cap or w.T
        for vb in w.v_bits:
            cache = tq.alloc_cache(w.B, w.H, t_cap, w.D, w.k_bits, vb, device=dev)
            torch.cuda.synchronize(dev)  # the cache's zero fill runs on torch's stream

            def enc_fn():
                tq.tq_encode_kv(k, v, w.k_bits, w.k_signed, vb, cache, stream=stream)

            def dec_fn():
                tq.tq_decode_kv(cache, w.T, w.k_bits, w.k_signed, vb, k_out=ko, v_out=vo, stream=stream)

            _time_launches(enc_fn, stream, 3)
            enc = _time_launches(enc_fn, stream, 10)
            dec = _time_launches(dec_fn, stream, 10)
            key = "%s_v%d" % (name, vb)
            if not (name == HEADLINE and vb == HEADLINE_V_BITS):
                out[key] = codec_roofline(name, vb, w.rows, w.D, w.k_bits, 1e3 * enc, 1e3 * dec, peak, peak_kind)
            if name == "long_context":
                # decode-step appends: one token per sequence at t_off = T + s (latency-bound)
                steps = [(a.to(dev), b.to(dev)) for a, b in make_append_steps(w)]
                g = torch.cuda.CUDAGraph()
                with torch.cuda.stream(stream):
                    for s_, (a, b) in enumerate(steps):
                        tq.tq_encode_kv(a, b, w.k_bits, w.k_signed, vb, cache, t_off=w.T + s_, stream=stream)
                torch.cuda.synchronize(dev)
                with torch.cuda.graph(g, stream=stream):
                    for s_, (a, b) in enumerate(steps):
                        tq.tq_encode_kv(a, b, w.k_bits, w.k_signed, vb, cache, t_off=w.T + s_, stream=stream)
                ms = _time_launches(g.replay, stream, 20)
                out["append_v%d" % vb] = {"us_per_step": r4(1e3 * ms / len(steps)), "rows_per_step": w.B * w.H,
                                          "steps_per_graph": len(steps)}
                if vb == 3:
                    out["batched_merge_v3"] = time_merge(tq, w, cache, t_cap, dev, stream, peak)
            out["attention_%s_v%d" % (name, vb)] = time_attention(tq, w, cache, t_cap, vb, dev, stream, peak,
                                                                  peak_kind)
            del cache
        del k, v, ko, vo
        torch.cuda.empty_cache()
    out["lloyd_max_fit"] = time_lloyd(tq, dev, stream)
    return out


def time_layers(tq, dev, stream, peak, peak_kind, rank):
    """The Llama-3-8B-shaped model: encode then decode of all 32 layers' KV
    for one 4096-token sequence, every layer with its own inputs, cache and
    outputs (1.28 GB, ten times the L2), as two CUDA graphs of 32 launches;
    CUDA events around each graph give the per-launch times."""
    from turboquant_kv_cache_tq_gb300.workloads import WORKLOADS, make_kv

    w = WORKLOADS["llama3_8b_layer"]
    kb, ks, vb = w.k_bits, w.k_signed, w.v_bits[0]
    B, H, T, D = w.B, w.H, w.T, w.D
    layers = []
    for i in range(LAYERS):
        k, v = make_kv(w, device=dev, seed=1000 * (rank + 1) + i)
        layers.append(dict(k=k, v=v, cache=tq.alloc_cache(B, H, T, D, kb, vb, device=dev),
                           ko=torch.empty_like(k), vo=torch.empty_like(v)))

    def enc_all():
        for L in layers:
            tq.tq_encode_kv(L["k"], L["v"], kb, ks, vb, L["cache"], stream=stream)

    def dec_all():
        for L in layers:
            tq.tq_decode_kv(L["cache"], T, kb, ks, vb, out_dtype=torch.bfloat16, k_out=L["ko"], v_out=L["vo"],
                            stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(2):
            enc_all()
            dec_all()
    torch.cuda.synchronize(dev)
    g_enc, g_dec = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_enc, stream=stream):
        enc_all()
    with torch.cuda.graph(g_dec, stream=stream):
        dec_all()
    reps = 50
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(reps)]
    with torch.cuda.stream(stream):
        for _ in range(5):
            g_enc.replay()
            g_dec.replay()
        for e in ev:
            e[0].record(stream)
            g_enc.replay()
            e[1].record(stream)
            g_dec.replay()
            e[2].record(stream)
    torch.cuda.synchronize(dev)
    enc_us = 1e3 * sum(e[0].elapsed_time(e[1]) for e in ev) / (reps * LAYERS)
    dec_us = 1e3 * sum(e[1].elapsed_time(e[2]) for e in ev) / (reps * LAYERS)
    step_ms = sum(e[0].elapsed_time(e[2]) for e in ev) / reps
    r = codec_roofline("llama3_8b_layer", vb, w.rows, D, kb, enc_us, dec_us, peak, peak_kind)
    r["tokens_per_s"] = r4(B * T * LAYERS / (step_ms / 1e3))
    r["layers_per_step"] = LAYERS
    del layers, g_enc, g_dec
    torch.cuda.empty_cache()
    return r


def time_attention(tq, w, cache, t_cap, vb, dev, stream, peak, peak_kind, G=4):
    """One decode step of fused attention over the whole packed cache of a
    workload (all t_cap tokens valid): 4 query heads per kv head (as in
    Llama-3-8B), one query token per sequence. Algorithmic bytes: the packed
    cache, read once."""
    g = torch.Generator(device=dev).manual_seed(6)
    q = torch.randn((w.B, w.H * G, 1, w.D), generator=g, device=dev).to(torch.bfloat16)
    out = torch.empty_like(q)
    ws_bytes = tq.tq_decode_attention_workspace_size(w.B, w.H, t_cap, w.D)
    work = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    ms = _time_launches(lambda: tq.tq_decode_attention(q, cache, t_cap, w.k_bits, w.k_signed, vb, out=out,
                                                       workspace=work, stream=stream), stream, 10)
    rows = w.B * w.H * t_cap
    per_row = w.D * w.k_bits // 8 + w.D * vb // 8 + 3 * (w.D // 32) * 2
    r = roofline_obj("attn_split_kernel", "%s_attention_v%d" % (w.name, vb), rows * per_row, 1e3 * ms, peak,
                     peak_kind)
    r["kv_tokens_per_s"] = r4(w.B * t_cap / (ms * 1e-3))
    r["query_heads"], r["kv_tokens"], r["launches"] = w.H * G, t_cap, 2
    return r


def time_merge(tq, w, cache, t_cap, dev, stream, peak):
    """Continuous batching: merge the cache's B rows, each with its own length
    (t_cap - 64 i tokens), into a fresh left-padded batch (mergeQuantRows).
    Bytes: every valid source token row read, the whole window written."""
    B = w.B
    lens = [t_cap - 64 * (i % 32) for i in range(B)]
    width = max(lens)
    rows = [({k: v[i:i + 1] for k, v in cache.items()}, n) for i, n in enumerate(lens)]
    dst = tq.alloc_cache(B, w.H, width, w.D, w.k_bits, cache["v_codes"].shape[-1] * 8 // w.D, device=dev)
    srcs = [(c, 0, 0, n) for c, n in rows]
    ms = _time_launches(lambda: tq.tq_cache_assemble(srcs, dst, width, stream=stream), stream, 10)
    per_tok = sum(t.shape[-1] * t.element_size() for t in cache.values()) * w.H
    nbytes = per_tok * (sum(lens) + B * width)
    return {"us": r4(1e3 * ms), "bytes_per_launch": nbytes, "GBps": r4(nbytes / (ms * 1e-3) / 1e9),
            "frac": r4(nbytes / (ms * 1e-3) / 1e9 / peak)}


def time_lloyd(tq, dev, stream, n=1 << 20, iters=500):
    """Lloyd-Max table fit (turboquant-tables.ts: 500 iterations on a
    unit-normal sample) of 2^20 samples at 4 and 8 bits, in microseconds per
    iteration: the 4 MB sample stays in L2 and every iteration is a chain of
    dependent steps ending in a grid barrier, so HBM bandwidth is not its
    bound. Its floor, measured here too: the same fit on an empty sample (an
    iteration is then its grid barrier, the cell-sum clearing and the means:
    barrier_floor_us) plus one pass over the sample at the L2's streaming
    rate (a 32 MB copy between buffers that stay in L2: l2_pass_us)."""
    g = torch.Generator(device=dev).manual_seed(7)
    x = torch.randn(n, generator=g, device=dev)
    out = {"samples": n, "iterations": iters}
    empty = torch.empty(0, device=dev)
    # the L2's streaming rate: a 32 MB copy between two buffers that stay in L2
    a = torch.empty(8 << 20, device=dev)
    b = torch.empty_like(a)
    l2_ms = _time_launches(lambda: b.copy_(a), stream, 50)
    l2_gbs = 2 * a.numel() * 4 / (l2_ms * 1e-3) / 1e9
    l2_pass = 4 * n / (l2_gbs * 1e9) * 1e3  # ms to read the sample once at that rate
    out["l2_GBps"] = r4(l2_gbs)
    out["l2_pass_us"] = r4(1e3 * l2_pass)
    for bits in (4, 8):
        K = 1 << bits
        init = torch.linspace(-3.0, 3.0, K, device=dev)
        work = torch.empty(tq.lib().tq_lloyd_max_fit_workspace_size(K), dtype=torch.uint8, device=dev)
        ms = _time_launches(lambda: tq.tq_lloyd_max_fit(x, init, iters, workspace=work, stream=stream), stream, 3)
        ms0 = _time_launches(lambda: tq.tq_lloyd_max_fit(empty, init, iters, workspace=work, stream=stream),
                             stream, 3)
        us, floor = 1e3 * ms / iters, 1e3 * ms0 / iters + 1e3 * l2_pass
        out["bits%d" % bits] = {"us_per_iteration": r4(us), "barrier_floor_us": r4(1e3 * ms0 / iters),
                                "floor_us": r4(floor), "frac_of_floor": r4(floor / us)}
    return out


def run_e2e(args, tq, units, kb, ks, vb, T, dev, stream):
    """Host buffers in, host buffers out, through the Python API. Every step
    copies each unit's K, V from pinned host memory, encodes and decodes it,
    and copies the decoded K, V back; units are pipelined over three streams
    (uploads, kernels, downloads) with per-unit events, so one unit's copies
    overlap other units' kernels and the two copy directions overlap each
    other. A device buffer is rewritten only after its previous reader is done
    (the next step's upload waits for the unit's encode, its decode for the
    unit's previous download)."""
    host_in = [(u["k"].cpu().pin_memory(), u["v"].cpu().pin_memory()) for u in units]
    host_out = [(torch.empty_like(a).pin_memory(), torch.empty_like(b).pin_memory()) for a, b in host_in]
    steps = max(1, min(args.steps, args.e2e_steps))
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    n = len(units)
    ev_in = [torch.cuda.Event() for _ in range(n)]
    ev_enc = [torch.cuda.Event() for _ in range(n)]
    ev_dec = [torch.cuda.Event() for _ in range(n)]
    ev_out = [torch.cuda.Event() for _ in range(n)]
    started = [False]

    def step():
        for i, (u, (hk, hv), (ok, ov)) in enumerate(zip(units, host_in, host_out)):
            with torch.cuda.stream(s_in):
                if started[0]:
                    s_in.wait_event(ev_enc[i])  # the previous step's encode has read the inputs
                u["k"].copy_(hk, non_blocking=True)
                u["v"].copy_(hv, non_blocking=True)
                ev_in[i].record(s_in)
            stream.wait_event(ev_in[i])
            tq.tq_encode_kv(u["k"], u["v"], kb, ks, vb, u["cache"], stream=stream)
            ev_enc[i].record(stream)
            if started[0]:
                stream.wait_event(ev_out[i])  # the previous step's download has read the outputs
            tq.tq_decode_kv(u["cache"], T, kb, ks, vb, out_dtype=torch.bfloat16, k_out=u["ko"], v_out=u["vo"],
                            stream=stream)
            ev_dec[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_dec[i])
                ok.copy_(u["ko"], non_blocking=True)
                ov.copy_(u["vo"], non_blocking=True)
                ev_out[i].record(s_out)
        started[0] = True

    def join():
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)

    step()
    join()
    torch.cuda.synchronize(dev)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_stream(stream)
    s_out.wait_stream(stream)
    for _ in range(steps):
        step()
    join()
    e1.record(stream)
    e1.synchronize()
    barrier()
    h2d = sum(a.numel() * a.element_size() + b.numel() * b.element_size() for a, b in host_in)
    d2h = sum(a.numel() * a.element_size() + b.numel() * b.element_size() for a, b in host_out)
    return {"ms": e0.elapsed_time(e1), "steps": steps, "h2d": h2d, "d2h": d2h}


def copy_floor(dev, reps: int):
    """Per-launch time of torch's device copy moving the bytes of one
    Llama-3-8B-shaped layer encode (11.67 MB read + 11.67 MB written), 32
    distinct buffers in one CUDA graph, the way the bench times the codec:
    what a plain memory-bound kernel reaches at this launch size; then the
    per-launch time of 32 one-element kernels, and of 32 codec launches on 8
    tokens of the layer shape (the codec's fixed cost per launch)."""
    n = 23330816 // 4  # int16 elements per copy
    srcs = [torch.zeros(n, dtype=torch.int16, device=dev) for _ in range(32)]
    dsts = [torch.empty_like(x) for x in srcs]
    s = torch.cuda.Stream(dev)

    def body():
        for a, b in zip(srcs, dsts):
            b.copy_(a)

    with torch.cuda.stream(s):
        body()
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        body()
    for _ in range(10):
        g.replay()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    with torch.cuda.stream(s):
        for _ in range(reps):
            g.replay()
    e1.record(s)
    e1.synchronize()
    us = 1e3 * e0.elapsed_time(e1) / reps / 32
    print("copy floor (32 x 11.67 MB copies in a CUDA graph): %.2f us per launch, %.0f GB/s" % (us, 23330816 / us / 1e3))
    # the launch floor: 32 launches of a one-element kernel in a CUDA graph
    tiny = [torch.zeros(1, device=dev) for _ in range(32)]
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        for t in tiny:
            t.add_(1.0)
    torch.cuda.synchronize(dev)
    with torch.cuda.graph(g2, stream=s):
        for t in tiny:
            t.add_(1.0)
    for _ in range(10):
        g2.replay()
    torch.cuda.synchronize(dev)
    e0.record(s)
    with torch.cuda.stream(s):
        for _ in range(reps):
            g2.replay()
    e1.record(s)
    e1.synchronize()
    print("launch floor (32 one-element kernels in a CUDA graph): %.2f us per launch"
          % (1e3 * e0.elapsed_time(e1) / reps / 32))
    # the codec's own fixed cost: 32 encode / decode launches of 8 tokens of
    # the layer shape (64 rows) in a CUDA graph
    import turboquant_kv_cache_tq_gb300 as tq

    layers = []
    for _ in range(32):
        k = torch.randn((1, 8, 8, 128), device=dev).to(torch.bfloat16)
        v = torch.randn((1, 8, 8, 128), device=dev).to(torch.bfloat16)
        layers.append((k, v, tq.alloc_cache(1, 8, 8, 128, 8, 3, device=dev), torch.empty_like(k), torch.empty_like(v)))

    def per_launch(fn):
        with torch.cuda.stream(s):
            fn()
        torch.cuda.synchronize(dev)
        g3 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g3, stream=s):
            fn()
        for _ in range(5):
            g3.replay()
        torch.cuda.synchronize(dev)
        e0.record(s)
        with torch.cuda.stream(s):
            for _ in range(reps):
                g3.replay()
        e1.record(s)
        e1.synchronize()
        return 1e3 * e0.elapsed_time(e1) / reps / 32

    enc = per_launch(lambda: [tq.tq_encode_kv(k, v, 8, True, 3, c, stream=s) for k, v, c, _, _ in layers])
    dec = per_launch(lambda: [tq.tq_decode_kv(c, 8, 8, True, 3, k_out=ko, v_out=vo, stream=s)
                              for _, _, c, ko, vo in layers])
    print("codec fixed cost (32 launches of 8 tokens x 8 kv heads in a CUDA graph): encode %.2f us, decode %.2f us "
          "per launch" % (enc, dec))


def host_link_floor(dev, reps: int):
    """The e2e step's copies alone: 32 layers' K, V (16.78 MB each layer) from
    pinned host memory to the device and the same bytes back, uploads and
    downloads on two streams at once, as run_e2e issues them; and each
    direction alone."""
    nb = 16777216 // 2
    hs = [torch.zeros(nb, dtype=torch.int16).pin_memory() for _ in range(32)]
    ho = [torch.empty(nb, dtype=torch.int16).pin_memory() for _ in range(32)]
    ds = [torch.empty(nb, dtype=torch.int16, device=dev) for _ in range(32)]
    do = [torch.zeros(nb, dtype=torch.int16, device=dev) for _ in range(32)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    total = 32 * nb * 2

    def timed(up: bool, down: bool) -> float:
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        main = torch.cuda.current_stream(dev)
        e0.record(main)
        s_in.wait_stream(main)
        s_out.wait_stream(main)
        for _ in range(reps):
            for i in range(32):
                if up:
                    with torch.cuda.stream(s_in):
                        ds[i].copy_(hs[i], non_blocking=True)
                if down:
                    with torch.cuda.stream(s_out):
                        ho[i].copy_(do[i], non_blocking=True)
        main.wait_stream(s_in)
        main.wait_stream(s_out)
        e1.record(main)
        e1.synchronize()
        return e0.elapsed_time(e1) / reps

    timed(True, True)
    for up, down, what in ((True, False, "host->device"), (False, True, "device->host"), (True, True, "both at once")):
        ms = timed(up, down)
        print("host link, %s: %.2f ms per 32 layers, %.0f GB/s per direction" % (what, ms, total / ms / 1e6))


def run_case(name: str, reps: int, v_bits=None, batch=None):
    """A small fixed case for profiling one kernel with ncu: the codec on one
    workload (encode then decode, `reps` times), one fused decode-attention
    step over the long-context cache shape, or the plain-copy floor of the
    Llama-3-8B-shaped layer ('copy_floor'), or the pinned host copies of the
    e2e step alone ('host_link'). Prints the median timing; it is not a bench
    line."""
    import turboquant_kv_cache_tq_gb300 as tq
    from turboquant_kv_cache_tq_gb300.workloads import WORKLOADS, make_kv

    dev = torch.device("cuda")
    if name == "copy_floor":
        copy_floor(dev, max(reps, 20))
        return
    if name == "host_link":
        host_link_floor(dev, max(reps, 3))
        return
    e = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(reps)]
    if name == "attention":
        B, H, T, D, G = 32 if batch is None else batch, 8, 8256, 128, 4
        vb = 3 if v_bits is None else v_bits
        cache = tq.alloc_cache(B, H, T, D, 8, vb, device=dev)
        g = torch.Generator(device=dev).manual_seed(0)
        for b0 in range(0, B, 4):  # encode in slices to keep the footprint small
            nb = min(4, B - b0)
            k = (0.5 * torch.randn((nb, H, T, D), generator=g, device=dev)).to(torch.bfloat16)
            v = (0.5 * torch.randn((nb, H, T, D), generator=g, device=dev)).to(torch.bfloat16)
            tq.tq_encode_kv(k, v, 8, True, vb, {n: t[b0:b0 + nb] for n, t in cache.items()})
            del k, v
        q = torch.randn((B, H * G, 1, D), generator=g, device=dev).to(torch.bfloat16)
        out = torch.empty_like(q)
        work = torch.empty(tq.tq_decode_attention_workspace_size(B, H, T, D), dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()
        for r in range(reps):
            e[r][0].record()
            tq.tq_decode_attention(q, cache, T, 8, True, vb, out=out, workspace=work)
            e[r][1].record()
        torch.cuda.synchronize()
        print("attention [%d,8,8256,128] k8s v%d: %.1f us" % (B, vb, _median_us(e)))
        return
    w = WORKLOADS[name]
    B = w.B if batch is None else batch
    k, v = make_kv(w, device=dev, B=B)
    vb = w.v_bits[0] if v_bits is None else v_bits
    cache = tq.alloc_cache(B, w.H, w.t_cap or w.T, w.D, w.k_bits, vb, device=dev)
    ko, vo = torch.empty_like(k), torch.empty_like(v)
    torch.cuda.synchronize()
    for r in range(reps):
        e[r][0].record()
        tq.tq_encode_kv(k, v, w.k_bits, w.k_signed, vb, cache)
        tq.tq_decode_kv(cache, w.T, w.k_bits, w.k_signed, vb, k_out=ko, v_out=vo)
        e[r][1].record()
    torch.cuda.synchronize()
    print("%s B=%d v%d encode+decode: %.1f us" % (name, B, vb, _median_us(e)))


def _median_us(events) -> float:
    return 1e3 * sorted(a.elapsed_time(b) for a, b in events)[len(events) // 2]


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-workloads", dest="workloads", action="store_false",
                    help="skip the secondary configurations")
    ap.add_argument("--no-cpu-all-cores", dest="cpu_all_cores", action="store_false",
                    help="skip the all-cores oracle timing")
    ap.add_argument("--case", default=None,
                    help="profiling aid: run one small case (a workload name, 'attention', 'copy_floor' or 'host_link') --reps times")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--v-bits", type=int, default=None, help="value bits of a --case workload")
    ap.add_argument("--batch", type=int, default=None, help="batch size of a --case workload (a smaller capture)")
    args = ap.parse_args(argv)
    if args.case:
        run_case(args.case, args.reps, args.v_bits, args.batch)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
