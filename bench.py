"""Benchmark of the DSA decode/prefill step on one GB300.

  python bench.py [--steps K] [--warmup W] [--workloads a,b,...]
  python bench.py --impl reference      # the CPU oracle as the reference arm
  python bench.py --stage S --workload X [--reps N]   # one stage, for profiler captures

One step = one pass of the whole path (indexer scores -> Top-K -> sparse MLA
attention) over one batch of seeded synthetic input through the C ABI
(dsa_decode_step).  By default every workload the metric is quoted on is
measured in one run: decode batch 1 (the headline line), decode batch 64,
long-context decode batch 4 and the 16384-token prefill.  For each:

* inputs are resident in HBM; R independent copies are rotated so that the bytes
  touched between two uses of a copy exceed twice the L2 cache;
* W untimed warm-up steps, then EXACTLY K timed steps (graph replays of R
  captured steps plus one graph of K mod R steps), CUDA events on the launching
  stream, synchronised on both sides;
* a sustained run of at least --min-seconds (whole graph replays, its step
  count reported as it is) so that the clock record covers a steady load;
* each stage alone (same rotation) for the roofline of the dominant kernel;
* end to end through the public call with pinned host buffers: the step's inputs
  host -> device and its outputs device -> host inside the timed region;
* the CPU oracle on a bounded sample of the same workload.

Prints one JSON line: the headline workload's numbers at the top level,
decode_tok_s / prefill_tok_s, and every workload under "workloads".
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "DSA layer decode tok/s & prefill tok/s on 1 GB300; % of HBM / tensor roofline"
HEADLINE = "decode_b1"
DEFAULT_WORKLOADS = ("decode_b1", "decode_b64", "decode_b4_long", "prefill_16k")
L2_BYTES = 129 * 1024 * 1024
DESCRIPTIONS = {
    "decode_b1": "decode batch 1: 1 query, ctx 32768, indexer 64x128 e4m3 + per-token fp32 scale, "
                 "top-k 2048, MLA 128 heads, bf16 latent 512+64, contiguous 64-token pages",
    "decode_b64": "decode batch 64: 1 query/seq, ctx ~ U{2048..8192}, shuffled 64-token pages, "
                  "indexer 64x128 e4m3, top-k 2048, MLA 128 heads, bf16 512+64",
    "decode_b4_long": "decode batch 4: ctx 131072 each, FP8 e4m3 latent (656-byte rows, per-token scale, "
                      "bf16 rope), indexer 64x128 e4m3, top-k 2048, MLA 128 heads",
    "prefill_16k": "prefill: 16384 causal tokens, indexer 64x128 e4m3, top-k 2048, MLA 128 heads, "
                   "bf16 512+64, inputs N(0,1) + rank-8 component",
    "decode_b64_mx": "decode batch 64 as decode_b64, indexer keys and queries MXFP8 (e4m3 codes, one E8M0 "
                     "scale per 32 elements, block magnitudes spread 2^-4..2^4)",
    "decode_b4_long_mx": "decode batch 4 as decode_b4_long, indexer keys and queries MXFP8 (e4m3 codes, one "
                         "E8M0 scale per 32 elements, block magnitudes spread 2^-4..2^4)",
    "decode_b4_long_t128": "decode batch 4 as decode_b4_long, FP8 latent rows with one power-of-two scale per "
                           "128 latent dims (tile magnitudes scaled by 2^{0,-1,-2})",
}
DEFAULT_STEPS = 200


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "src": "fallback"}


def measure_fp8_peak(torch, dev):
    """Dense e4m3 x e4m3 -> bf16 GEMM throughput of the vendor library at
    8192^3 (torch._scaled_mm, the library path), best of 10 after warm-up,
    with and without fast accumulation; returns the larger (TFLOP/s) and how."""
    n = 8192
    try:
        a = torch.randn((n, n), device=dev).to(torch.float8_e4m3fn)
        b = torch.randn((n, n), device=dev).to(torch.float8_e4m3fn).t()    # column-major operand
        one = torch.ones((), device=dev, dtype=torch.float32)
        best = {}
        for fast in (False, True):
            for _ in range(3):
                torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16, use_fast_accum=fast)
            times = []
            for _ in range(10):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16, use_fast_accum=fast)
                e1.record()
                torch.cuda.synchronize()
                times.append(e0.elapsed_time(e1) / 1e3)
            best[fast] = 2.0 * n ** 3 / min(times) / 1e12
        del a, b
        torch.cuda.empty_cache()
        v = max(best.values())
        return v, (f"torch._scaled_mm e4m3 {n}^3 -> bf16, best of 10 (fp32 accumulate {best[False]:.0f}, "
                   f"fast accumulate {best[True]:.0f} TFLOP/s; the larger is the peak)")
    except Exception as e:   # a library without this path: the nominal ratio to the measured BF16 peak
        return None, f"torch._scaled_mm unavailable ({type(e).__name__}); 2 x measured BF16 (nominal ratio)"


# ----------------------------------------------------------------------------- bytes / flops

def algorithmic(wl):
    """What each stage must move (bytes) or compute (flops) for this workload."""
    import numpy as np
    n = wl.q_pos.astype(np.int64) + 1
    m = np.minimum(n, wl.K)
    # keys shared by the queries of a sequence are read once
    per_seq = {}
    for b, nn in zip(wl.q_seq, n):
        per_seq[int(b)] = max(per_seq.get(int(b), 0), int(nn))
    scale_bytes = wl.D_I // 32 if wl.idx_dtype == "mx_e4m3" else 4   # per key / per query head
    key_bytes = sum(per_seq.values()) * (wl.D_I + scale_bytes)
    qi_bytes = wl.T * wl.H_I * (wl.D_I + scale_bytes + 4)
    score_bytes = int(n.sum()) * 4
    row_b = 656 if wl.mla_dtype in ("e4m3", "e4m3_t128") else wl.d_qk * 2
    gather = int(m.sum()) * row_b
    q_bytes = wl.T * wl.H * wl.d_qk * 2
    out_bytes = wl.T * wl.H * (wl.d_v * 2 + 4)
    idx_bytes = wl.T * wl.K * 4
    causal_pairs = int(n.sum())
    return {
        "indexer": {"bytes": key_bytes + qi_bytes + score_bytes,
                    "flops": causal_pairs * wl.H_I * wl.D_I * 2},
        "topk": {"bytes": score_bytes + idx_bytes},
        "attn": {"bytes": gather + q_bytes + out_bytes + idx_bytes,
                 "flops": int(m.sum()) * wl.H * (wl.d_qk + wl.d_v) * 2},
        # the step: keys + indexer queries + gathered rows + MLA queries + outputs
        "step_bytes": key_bytes + qi_bytes + gather + q_bytes + out_bytes,
        "cache_bytes": wl.cache_rows * (wl.D_I + scale_bytes + wl.row_bytes),
    }


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampled every 50 ms (read only); samples are kept with their
    time stamps so that the ones inside the timed windows can be picked out."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.proc, self.windows, self.lines = index, None, [], []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.15)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            self.lines = [l for l in out.splitlines() if l.strip()]

    def window(self, t0: float, t1: float):
        self.windows.append((t0, t1))

    def summary(self):
        sm, mx, reasons, n_all = [], None, set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                clk, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            n_all += 1
            if not any(a - 0.06 <= ts <= b + 0.06 for a, b in self.windows):
                continue
            sm.append(clk)
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples_under_load": len(sm), "samples": n_all,
                "window_s": round(sum(b - a for a, b in self.windows), 3)}


# ----------------------------------------------------------------------------- helpers

def kernel_count(plan: str) -> int:
    return sum(plan.count(k) for k in ("indexer_tc", "indexer_generic", "topk_radix", "topk_fused", "attn_tc",
                                       "attn_generic", "attn_combine", "prolog_proj", "prolog_epilogue"))


def traffic_from_profiles(kernel_file: str, workload: str):
    """DRAM bytes per launch recorded in profiles/ for this workload, if the
    kernel source is unchanged since the capture (sha256 prefix)."""
    src = os.path.join(ROOT, "dsa_indexed_sparse_gb300", "csrc", kernel_file)
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    for f in sorted(os.listdir(pdir)):
        if not f.endswith(".md"):
            continue
        for line in open(os.path.join(pdir, f)):
            mt = re.match(r"traffic_per_launch:\s*workload=(\S+)\s+kernel_src=(\S+)\s+sha=(\w+)\s+bytes=(\d+)", line)
            if mt and mt.group(1) == workload and mt.group(2) == kernel_file and mt.group(3) == sha:
                return int(mt.group(4))
    return None


def time_replays(torch, graphs, stream):
    """Replays the graphs in order on `stream` (the stream the events are
    recorded on); returns seconds and the host window."""
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    h0 = time.time()
    with torch.cuda.stream(stream):
        start.record(stream)
        for g in graphs:
            g.replay()
        end.record(stream)
    torch.cuda.synchronize()
    h1 = time.time()
    return start.elapsed_time(end) / 1e3, (h0, h1)


def capture(torch, fn, items, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for c in items:
            fn(c)  # warm: attribute setup happens outside capture
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for c in items:
                fn(c)
    return g


# ----------------------------------------------------------------------------- CPU oracle leg

def oracle_rate(wl, budget_s: float):
    """The CPU oracle as it stands on a bounded sample of the workload: whole
    decode steps (all queries) for decode workloads; a subset of query rows for
    prefill.  Returns (tokens/s, sample description)."""
    from oracle import dsa_oracle as O
    t0 = time.perf_counter()
    if wl.name.startswith("prefill"):
        import numpy as np
        rows = list(np.linspace(0, wl.T - 1, 8).astype(int))
        done = 0
        while True:
            O.decode_step(wl, ts=rows)
            done += len(rows)
            if time.perf_counter() - t0 > budget_s:
                break
        el = time.perf_counter() - t0
        return done / el, (f"{done} query rows of the prefill (8 rows spread over positions 0..{wl.T - 1}, "
                           f"their mean cost stands for the whole step: extrapolated) in {el:.1f} s")
    steps = 0
    while True:
        O.decode_step(wl)
        steps += 1
        if time.perf_counter() - t0 > budget_s:
            break
    el = time.perf_counter() - t0
    return steps * wl.T / el, f"{steps} full decode steps ({steps * wl.T} query tokens) in {el:.1f} s"


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# ----------------------------------------------------------------------------- profiling mode

def profile_stage(torch, dsa, W, wl, dev, stage, reps):
    """Runs one stage `reps` times on one copy of the workload (its inputs made by
    the stages before it), for profiler captures of a single kernel."""
    d = W.device_tensors(wl, dev)
    seq, idxr, mla = dsa.Seq(**d["seq"]), dsa.Indexer(**d["indexer"]), dsa.Mla(**d["mla"])
    ld = (wl.max_ctx + 3) // 4 * 4
    scores = torch.empty((wl.T, ld), dtype=torch.float32, device=dev)
    sel = torch.empty((wl.T, wl.K), dtype=torch.int32, device=dev)
    out = torch.empty((wl.T, wl.H, wl.d_v), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((wl.T, wl.H), dtype=torch.float32, device=dev)
    attn_ws = torch.empty(max(16, dsa.sparse_mla_attn_workspace_size(seq, mla, wl.K)), dtype=torch.uint8, device=dev)
    ws = torch.empty(dsa.decode_workspace_size(seq, idxr, mla, wl.K), dtype=torch.uint8, device=dev)
    fns = {"indexer": lambda: dsa.indexer_scores(seq, idxr, scores),
           "topk": lambda: dsa.topk(seq, scores, wl.K, sel),
           "attn": lambda: dsa.sparse_mla_attn(seq, mla, sel, wl.K, out, lse=lse, workspace=attn_ws),
           "step": lambda: dsa.decode_step(seq, idxr, mla, wl.K, out, ws, lse=lse)}
    for name in ("indexer", "topk", "attn"):   # the inputs of the profiled stage
        fns[name]()
    torch.cuda.synchronize()
    for _ in range(reps):
        fns[stage]()
    torch.cuda.synchronize()
    dsa.check_status()
    print(f"profiled {stage} x{reps} on {wl.name}: {dsa.last_plan()}")
    return 0


# ----------------------------------------------------------------------------- one workload

def measure_workload(torch, np, dsa, W, name, steps, warmup, min_seconds, peaks, dev, clk, oracle_seconds):
    wl = W.make(name, seed=0)
    alg = algorithmic(wl)
    # copies: the bytes a step touches, times the copies rotated, exceed 2 x L2;
    # bounded by memory (the caches of one copy)
    copies_n = max(1, math.ceil(2 * L2_BYTES / max(alg["step_bytes"], 1)) + 1)
    copies_n = min(copies_n, 64, max(1, int(24e9 // max(alg["cache_bytes"], 1))))
    tens = W.device_tensors(wl, dev, copies=copies_n) if copies_n > 1 else [W.device_tensors(wl, dev)]
    runs = []
    for d in tens:
        seq, idxr, mla = dsa.Seq(**d["seq"]), dsa.Indexer(**d["indexer"]), dsa.Mla(**d["mla"])
        out = torch.empty((wl.T, wl.H, wl.d_v), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((wl.T, wl.H), dtype=torch.float32, device=dev)
        runs.append(dict(seq=seq, idxr=idxr, mla=mla, out=out, lse=lse))
    R = len(runs)
    ws_bytes = dsa.decode_workspace_size(runs[0]["seq"], runs[0]["idxr"], runs[0]["mla"], wl.K)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    ld = (wl.max_ctx + 3) // 4 * 4
    scores = torch.empty((wl.T, ld), dtype=torch.float32, device=dev)
    sel = torch.empty((wl.T, wl.K), dtype=torch.int32, device=dev)
    attn_ws = torch.empty(max(16, dsa.sparse_mla_attn_workspace_size(runs[0]["seq"], runs[0]["mla"], wl.K)),
                          dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream()

    def step(r):
        dsa.decode_step(r["seq"], r["idxr"], r["mla"], wl.K, r["out"], ws, lse=r["lse"], stream=stream)

    def st_indexer(r):
        dsa.indexer_scores(r["seq"], r["idxr"], scores, stream=stream)

    def st_topk(r):
        dsa.topk(r["seq"], scores, wl.K, sel, stream=stream)

    def st_attn(r):
        dsa.sparse_mla_attn(r["seq"], r["mla"], sel, wl.K, r["out"], lse=r["lse"], workspace=attn_ws, stream=stream)

    # the configuration runs clean before anything is timed
    with torch.cuda.stream(stream):
        step(runs[0])
    plan = dsa.last_plan()
    dsa.check_status(stream)

    g_full = capture(torch, step, runs, stream)
    g_rem = capture(torch, step, runs[:steps % R], stream) if steps % R else None
    # warm-up: at least `warmup` untimed steps
    with torch.cuda.stream(stream):
        for _ in range(max(1, math.ceil(warmup / R))):
            g_full.replay()
    torch.cuda.synchronize()
    # exactly `steps` timed steps
    seq_graphs = [g_full] * (steps // R) + ([g_rem] if g_rem is not None else [])
    t_step, win = time_replays(torch, seq_graphs, stream)
    clk.window(*win)
    dsa.check_status(stream)
    ms_per_step = 1e3 * t_step / steps
    value = wl.T * steps / t_step

    # sustained: whole replays for at least min_seconds (clock record under steady load)
    n_rep = max(1, math.ceil(min_seconds / max(t_step / steps * R, 1e-9)))
    t_sus, win = time_replays(torch, [g_full] * n_rep, stream)
    clk.window(*win)
    dsa.check_status(stream)
    sustained = {"steps": n_rep * R, "seconds": t_sus, "ms_per_step": 1e3 * t_sus / (n_rep * R),
                 "tok_s": wl.T * n_rep * R / t_sus}
    del g_full, g_rem

    # each stage alone over the same rotation (>= 200 steps or 50 ms)
    stage_t, stage_plan = {}, {}
    for sname, fn in (("indexer", st_indexer), ("topk", st_topk), ("attn", st_attn)):
        with torch.cuda.stream(stream):
            fn(runs[0])
        stage_plan[sname] = dsa.last_plan()
        g = capture(torch, fn, runs, stream)
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        t1, _ = time_replays(torch, [g], stream)
        rp = max(1, min(2000, max(math.ceil(200 / R), math.ceil(0.05 / max(t1, 1e-9)))))
        tt, win = time_replays(torch, [g] * rp, stream)
        clk.window(*win)
        stage_t[sname] = tt / (rp * R)
        dsa.check_status(stream)
        del g
    dom = max(stage_t, key=stage_t.get)
    prefill = wl.name.startswith("prefill")
    kernels = {}
    for sname in stage_t:
        if prefill and sname in ("indexer", "attn"):
            if sname == "indexer":
                pk, psrc = peaks["fp8_tflops"], peaks["fp8_src"]
            else:
                pk, psrc = peaks["bf16_tflops"], "measured bf16 burst"
            ach = alg[sname]["flops"] / stage_t[sname] / 1e12
            kernels[sname] = {"bound": "tensor", "achieved": ach, "peak": pk, "unit": "TFLOP/s",
                              "frac": ach / pk, "peak_src": psrc}
        else:
            ach = alg[sname]["bytes"] / stage_t[sname] / 1e9
            kernels[sname] = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                              "frac": ach / peaks["hbm_gbs"], "peak_src": peaks["src"] + " hbm copy"}
        kfile = {"indexer": "indexer.cu", "topk": "topk.cu", "attn": "attn.cu"}[sname]
        kernels[sname]["traffic"] = traffic_from_profiles(kfile, name)
        kernels[sname]["kernel"] = stage_plan[sname]
        kernels[sname]["us"] = stage_t[sname] * 1e6
    roof = dict(kernels[dom])
    roof["stage"] = dom

    # end to end through the public call with host buffers (pinned): the step's
    # inputs (indexer query + scales + head weights, MLA query, positions; for a
    # prefill also the caches its tokens fill) host -> device in one packed
    # buffer, out + lse back in another, exactly `steps` steps.  Pipelined as a
    # serving loop runs it: NS device buffer sets; later steps' inputs go in on a
    # copy stream while step i computes, step i's results come back on another.
    # Every step's copies are inside the timed region; a slot's buffers are reused
    # only after the copies and the step that used them NS steps earlier are done
    # (three sets give each slot's copies a whole step of slack: at prefill size
    # the two directions' copies take about as long as the step's compute).
    r0 = runs[0]
    parts = [r0["idxr"].q, r0["idxr"].q_scale, r0["idxr"].w, r0["mla"].q, r0["seq"].q_pos, r0["seq"].q_seq]
    if prefill:
        parts += [r0["idxr"].k_cache, r0["idxr"].k_scale, r0["mla"].kv_cache]
    sizes = [t.numel() * t.element_size() for t in parts]
    offs = np.cumsum([0] + [(s + 255) // 256 * 256 for s in sizes])
    h_pack = torch.empty(int(offs[-1]), dtype=torch.uint8).pin_memory()
    for t, o, n in zip(parts, offs[:-1], sizes):
        h_pack[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())
    out_bytes = r0["out"].numel() * 2
    NS = 3
    slots = []
    for _ in range(NS):
        d_pack = torch.empty(int(offs[-1]), dtype=torch.uint8, device=dev)
        views = [d_pack[o:o + n].view(t.dtype).view(t.shape) for t, o, n in zip(parts, offs[:-1], sizes)]
        kc, ks, kv = (views[6], views[7], views[8]) if prefill else (r0["idxr"].k_cache, r0["idxr"].k_scale,
                                                                     r0["mla"].kv_cache)
        e_seq = dsa.Seq(q_seq=views[5], q_pos=views[4], block_table=r0["seq"].block_table,
                        max_ctx=r0["seq"].max_ctx, cache_rows=r0["seq"].cache_rows, page_size=r0["seq"].page_size,
                        q_per_seq=r0["seq"].q_per_seq)
        e_idx = dsa.Indexer(q=views[0], w=views[2], k_cache=kc, q_scale=views[1], k_scale=ks,
                            dtype=r0["idxr"].dtype)
        e_mla = dsa.Mla(q=views[3], kv_cache=kv, d_latent=wl.d_latent, d_rope=wl.d_rope,
                        softmax_scale=wl.softmax_scale, dtype=r0["mla"].dtype)
        d_res = torch.empty(out_bytes + r0["lse"].numel() * 4, dtype=torch.uint8, device=dev)
        slots.append(dict(pack=d_pack, seq=e_seq, idx=e_idx, mla=e_mla, res=d_res,
                          out=d_res[:out_bytes].view(torch.bfloat16).view(r0["out"].shape),
                          lse=d_res[out_bytes:].view(torch.float32).view(r0["lse"].shape),
                          h_res=torch.empty(d_res.numel(), dtype=torch.uint8).pin_memory(),
                          loaded=torch.cuda.Event(), computed=torch.cuda.Event(), returned=torch.cuda.Event()))
    h2d = int(sum(sizes))
    d2h = int(slots[0]["res"].numel())
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_step(i):
        sl = slots[i % NS]
        if i >= NS:
            s_in.wait_event(sl["computed"])      # the step NS back has read this slot's inputs
        with torch.cuda.stream(s_in):
            sl["pack"].copy_(h_pack, non_blocking=True)
            sl["loaded"].record(s_in)
        stream.wait_event(sl["loaded"])
        if i >= NS:
            stream.wait_event(sl["returned"])    # its results from NS steps back are on the host
        with torch.cuda.stream(stream):
            dsa.decode_step(sl["seq"], sl["idx"], sl["mla"], wl.K, sl["out"], ws, lse=sl["lse"], stream=stream)
            sl["computed"].record(stream)
        s_out.wait_event(sl["computed"])
        with torch.cuda.stream(s_out):
            sl["h_res"].copy_(sl["res"], non_blocking=True)
            sl["returned"].record(s_out)

    for i in range(max(3, min(warmup, 20))):
        e2e_step(i)
    torch.cuda.synchronize()

    # n pipelined steps captured in one CUDA graph (the copy streams forked from
    # and joined back into the capturing stream), as the device-side steps are:
    # replays then cost no host time per step.  Replays run in stream order, so a
    # replay's first NS steps find their slots free.  Each replay fills and drains
    # the pipeline (its first step's inputs and its last step's results cross alone),
    # so up to 400 steps go into one graph: one fill and drain per timed run, as in
    # a serving loop that runs on.
    def capture_e2e(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fork = torch.cuda.Event()
            fork.record(stream)
            s_in.wait_event(fork)
            s_out.wait_event(fork)
            for i in range(n):
                e2e_step(i)
            for k in range(min(n, NS)):
                stream.wait_event(slots[(n - 1 - k) % NS]["returned"])
        return g

    E = min(steps, 400)
    g_e2e = capture_e2e(E)
    g_e2e_rem = capture_e2e(steps % E) if steps % E else None
    with torch.cuda.stream(stream):
        g_e2e.replay()
    torch.cuda.synchronize()
    t_e2e, win = time_replays(torch, [g_e2e] * (steps // E) + ([g_e2e_rem] if g_e2e_rem else []), stream)
    clk.window(*win)
    del g_e2e, g_e2e_rem
    e2e = {"value": wl.T * steps / t_e2e, "unit": "tok/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": 1e3 * t_e2e / steps,
           "pipeline": f"{NS} buffer sets: inputs in on a copy stream while earlier steps compute, results "
                       f"out on another; {E} steps per CUDA graph replay; every step's copies inside the timed "
                       f"region"}
    dsa.check_status(stream)

    res = {
        "workload": f"{name}: {DESCRIPTIONS[name]}",
        "tok_s": value, "ms_per_step": ms_per_step, "steps": steps, "warmup": warmup,
        "sustained": sustained,
        "plan": plan,
        "l2": f"{R} rotated input copies, {alg['step_bytes'] / 1e6:.1f} MB touched per step "
              f"(inputs larger than L2 between reuses)",
        "cuda_graph": f"{R} steps per graph replay",
        "step_algorithmic_bytes": alg["step_bytes"],
        "step_hbm_frac": alg["step_bytes"] / (ms_per_step / 1e3) / 1e9 / peaks["hbm_gbs"],
        "stage_us": {k: v * 1e6 for k, v in stage_t.items()},
        "roofline": roof,
        "kernels": kernels,
        "e2e": e2e,
        "gpu_launches": kernel_count(plan) * steps,
    }
    del runs, tens, ws, scores, sel, attn_ws, h_pack, slots
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    if oracle_seconds > 0:
        rate, sample = oracle_rate(wl, oracle_seconds)
        res["cpu_baseline"] = {"value": rate, "unit": "tok/s", "cores": host_cores(), "kind": "oracle",
                               "sample": sample}
    return res


# ----------------------------------------------------------------------------- the indexer prolog

def measure_prolog(torch, dsa, W, name, steps, warmup, peaks, dev, clk):
    """dsa_indexer_prolog on one batch of new tokens: exactly `steps` timed calls
    over rotated input copies (graph replays), with the roofline of the
    projection: weights + inputs + outputs against HBM for a decode batch, the
    projections' flops against the BF16 peak for a prefill batch."""
    pl = W.make_prolog(name, seed=0)
    HD = pl.H_I * pl.D_I
    w_bytes = 2 * (HD * pl.d_q + (pl.D_I + pl.H_I) * pl.d_model)
    in_bytes = 2 * pl.T * (pl.d_model + pl.d_q)
    out_bytes = pl.T * (HD + 4 * pl.H_I + 4 * pl.H_I + pl.D_I + 4)
    flops = 2 * pl.T * (HD * pl.d_q + (pl.D_I + pl.H_I) * pl.d_model)
    step_bytes = w_bytes + in_bytes + out_bytes
    R = max(1, min(16, math.ceil(2 * L2_BYTES / step_bytes) + 1))
    stream = torch.cuda.Stream()
    runs = []
    for _ in range(R):
        d = W.prolog_device_tensors(pl, dev)
        seq, pro = dsa.Seq(**d["seq"]), dsa.Prolog(**d["prolog"])
        runs.append(dict(seq=seq, pro=pro, k_cache=d["k_cache"], k_scale=d["k_scale"],
                         q=torch.empty((pl.T, pl.H_I, pl.D_I), dtype=torch.uint8, device=dev),
                         qs=torch.empty((pl.T, pl.H_I), dtype=torch.float32, device=dev),
                         w=torch.empty((pl.T, pl.H_I), dtype=torch.float32, device=dev)))
    ws = torch.empty(dsa.indexer_prolog_workspace_size(runs[0]["seq"], runs[0]["pro"]), dtype=torch.uint8, device=dev)

    def call(r):
        dsa.indexer_prolog(r["seq"], r["pro"], r["q"], r["qs"], r["w"], r["k_cache"], r["k_scale"], ws, stream=stream)

    with torch.cuda.stream(stream):
        call(runs[0])
    plan = dsa.last_plan()
    dsa.check_status(stream)
    g_full = capture(torch, call, runs, stream)
    g_rem = capture(torch, call, runs[:steps % R], stream) if steps % R else None
    with torch.cuda.stream(stream):
        for _ in range(max(1, math.ceil(warmup / R))):
            g_full.replay()
    torch.cuda.synchronize()
    t, win = time_replays(torch, [g_full] * (steps // R) + ([g_rem] if g_rem is not None else []), stream)
    clk.window(*win)
    dsa.check_status(stream)
    us = 1e6 * t / steps
    if pl.T >= 1024:
        ach = flops / (us * 1e-6) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": ach / peaks["bf16_tflops"], "peak_src": "measured bf16 burst"}
    else:
        ach = step_bytes / (us * 1e-6) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"], "peak_src": peaks["src"] + " hbm copy"}
    roof["traffic"] = traffic_from_profiles("prolog.cu", name)
    res = {"workload": f"{name}: {pl.T} new tokens, hidden {pl.d_model}, query latent {pl.d_q}, "
                       f"indexer {pl.H_I}x{pl.D_I}; bf16 inputs and weights",
           "us_per_call": us, "tok_s": pl.T / (us * 1e-6), "steps": steps, "plan": plan,
           "algorithmic_bytes": step_bytes, "flops": flops, "roofline": roof,
           "l2": f"{R} rotated input copies"}
    del runs, ws, g_full, g_rem
    torch.cuda.empty_cache()
    return res


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=DEFAULT_STEPS)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workloads", default=",".join(DEFAULT_WORKLOADS),
                    help="comma-separated workloads; the first is the headline line")
    ap.add_argument("--workload", default=None,
                    help="one workload only (also the workload of --stage and --impl reference)")
    ap.add_argument("--min-seconds", type=float, default=0.25,
                    help="length of the sustained run per workload")
    ap.add_argument("--oracle-seconds", type=float, default=8.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prolog", action="store_true", help="skip the indexer-prolog measurement")
    ap.add_argument("--stage", choices=["indexer", "topk", "attn", "step", "prolog"], default=None,
                    help="profiling mode: run this stage --reps times on one input copy and exit "
                         "(no timing, no JSON line); for ncu captures")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--prefill-len", type=int, default=None,
                    help="profiling mode only: run the prefill recipe at this many tokens (a small "
                         "case of the same kernels for profiler captures)")
    args = ap.parse_args()
    if args.steps < 1:
        ap.error("--steps must be >= 1")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    import dsa_workloads as W
    names = [args.workload] if args.workload else [s for s in args.workloads.split(",") if s]
    for nm in names:
        if nm not in DESCRIPTIONS and not (args.stage == "prolog" and nm in W.PROLOG_SPECS):
            ap.error(f"unknown workload {nm}")

    if args.impl == "reference":
        if rank != 0:
            return 0
        wl = W.make(names[0], seed=0)
        steps = args.steps
        # each step a bounded sample of the workload: about 2 s of oracle work
        for _ in range(min(max(args.warmup, 0), 1)):
            oracle_rate(wl, 0.0)
        budget = max(1.0, min(120.0, 2.0 * steps))
        rate, sample = oracle_rate(wl, budget)
        unit = "tok/s"
        line = {"impl": "reference", "metric": METRIC, "value": rate, "unit": unit, "n_gpus": 1,
                "steps": steps, "warmup": args.warmup, "ms_per_step": 1e3 * wl.T / rate,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": {"workload": f"{names[0]}: {DESCRIPTIONS[names[0]]}"},
                "cpu_baseline": {"value": rate, "unit": unit, "cores": host_cores(), "kind": "oracle",
                                 "sample": sample},
                "e2e": {"value": rate, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return 0

    if world > 1 or args.gpus != 1:
        print(json.dumps({"error": "single-GPU path: the benchmark runs on one GPU (replicas only)"}))
        return 2

    import numpy as np
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import dsa_indexed_sparse_gb300 as dsa

    peaks = load_peaks()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    if args.stage == "prolog":
        # profiling mode for the indexer prolog: --reps calls on one input copy
        nm = args.workload if args.workload in W.PROLOG_SPECS else "prolog_decode_b64"
        pl = W.make_prolog(nm, seed=0)
        d = W.prolog_device_tensors(pl, dev)
        seq, pro = dsa.Seq(**d["seq"]), dsa.Prolog(**d["prolog"])
        q = torch.empty((pl.T, pl.H_I, pl.D_I), dtype=torch.uint8, device=dev)
        qs = torch.empty((pl.T, pl.H_I), dtype=torch.float32, device=dev)
        w = torch.empty((pl.T, pl.H_I), dtype=torch.float32, device=dev)
        ws = torch.empty(dsa.indexer_prolog_workspace_size(seq, pro), dtype=torch.uint8, device=dev)
        for _ in range(args.reps):
            dsa.indexer_prolog(seq, pro, q, qs, w, d["k_cache"], d["k_scale"], ws)
        torch.cuda.synchronize()
        dsa.check_status()
        print(f"profiled prolog x{args.reps} on {nm}: {dsa.last_plan()}")
        return 0
    if args.stage:
        nm = names[0]
        if args.prefill_len is not None:
            if nm != "prefill_16k":
                ap.error("--prefill-len needs --workload prefill_16k")
            wl = W.make(nm, seed=0, ctx=[args.prefill_len], q_len=args.prefill_len)
        else:
            wl = W.make(nm, seed=0)
        return profile_stage(torch, dsa, W, wl, dev, args.stage, args.reps)

    warmup = max(3, args.warmup)
    fp8, fp8_src = measure_fp8_peak(torch, dev)
    peaks["fp8_tflops"] = fp8 if fp8 else 2.0 * peaks["bf16_tflops"]
    peaks["fp8_src"] = ("measured: " if fp8 else "") + fp8_src
    oracle_s = 0.0 if args.no_cpu_baseline else args.oracle_seconds
    results = {}
    with ClockSampler(0) as clk:
        for nm in names:
            results[nm] = measure_workload(torch, np, dsa, W, nm, args.steps, warmup, args.min_seconds, peaks, dev,
                                           clk, 0.0)
        prolog = {} if args.no_prolog or args.workload else {
            nm: measure_prolog(torch, dsa, W, nm, args.steps, warmup, peaks, dev, clk)
            for nm in ("prolog_decode_b64", "prolog_prefill_4k")}
    clocks = clk.summary()
    # the CPU oracle after the GPU work (host cores only; not inside any timed window)
    if oracle_s > 0:
        for nm in names:
            wl = W.make(nm, seed=0)
            rate, sample = oracle_rate(wl, oracle_s)
            results[nm]["cpu_baseline"] = {"value": rate, "unit": "tok/s", "cores": host_cores(), "kind": "oracle",
                                           "sample": sample}
    head = results[names[0]]
    dec = next((results[n] for n in names if n.startswith("decode")), None)
    pre = next((results[n] for n in names if n.startswith("prefill")), None)
    line = {
        "metric": METRIC, "value": head["tok_s"], "unit": "tok/s", "n_gpus": 1, "steps": args.steps,
        "warmup": warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3+bf16 (fp32 accumulate)", "data": "synthetic",
        "decode_tok_s": dec["tok_s"] if dec else None,
        "prefill_tok_s": pre["tok_s"] if pre else None,
        "config": {"workload": head["workload"], "l2": head["l2"], "cuda_graph": head["cuda_graph"],
                   "plan": head["plan"], "step_algorithmic_bytes": head["step_algorithmic_bytes"],
                   "step_hbm_frac": head["step_hbm_frac"], "stage_us": head["stage_us"],
                   "sustained": head["sustained"]},
        "roofline": head["roofline"],
        "e2e": head["e2e"],
        "gpu_launches": head["gpu_launches"],
        "clocks": clocks,
        "peaks": {k: peaks[k] for k in ("hbm_gbs", "bf16_tflops", "fp8_tflops", "fp8_src", "src")},
        "workloads": results,
        "prolog": prolog,
    }
    if "cpu_baseline" in head:
        line["cpu_baseline"] = head["cpu_baseline"]
    print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
