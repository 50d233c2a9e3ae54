#!/usr/bin/env python3
"""Benchmark of the causal GQA attention step on GB300.

One step = the whole path for one packed batch: qkv split + Q/K RMSNorm +
RoPE + cache append (prologue kernel; for prefill it also writes the prepared
Q) and causal GQA attention (tcgen05 prefill kernel; split-KV + combine for
decode, which prepares its few Q rows itself).

Headline (``value``): prefill TFLOP/s of the whole step on the largest
single-GPU workload, one 32 768-token sequence with Hq 64 / Hkv 8 / D 128
(``long_prefill_T32768_hq64_hkv8``).  FLOPs = 4 * D * Hq * (unmasked
query-key pairs, diagonal included).  Every other workload is measured in the
same run under its own key: the Qwen3-4B-shaped prefill (8 packed sequences,
lengths U[256, 2048]), the 64-request decode batch (KV-read GB/s, the decode
half of the metric), both over bf16 and one-byte E4M3 caches, the mixed
prefill-chunk + decode step, the attention layer with its Q/K/V and output
projections (Qwen3-4B hidden size 2560), the tiny 12-token workload
(microseconds per call) and token sampling.  Inputs are seeded synthetic tensors resident in
HBM; L2 is flushed before every timed step, outside the timed events: a
256 MiB buffer is written, then another 256 MiB buffer is read, so that the
step starts with none of its inputs in L2 and with no dirty lines of the flush
left for it to write back.

``--impl reference`` times the CPU fp64 oracle on the host cores instead
(a bounded sample of the same workload per step).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefill attn TFLOP/s & decode KV-read GB/s on 1 GB300, % of roofline"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


ONLY_PARTS = ("long_prefill", "prefill", "prefill_e4m3", "decode", "decode_e4m3", "mixed", "projection",
              "sampling", "tiny")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="long_prefill_T32768_hq64_hkv8")
    ap.add_argument("--prefill-workload", default="qwen3_4b_prefill_8seq_U256_2048",
                    help="second prefill workload, reported under its own key")
    ap.add_argument("--decode-workload", default="decode_b64_cache_U512_8192")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode measurement")
    ap.add_argument("--mixed-workload", default="mixed_4x1024chunks_256decode")
    ap.add_argument("--no-mixed", action="store_true", help="skip the mixed-step measurement")
    ap.add_argument("--no-sampling", action="store_true", help="skip the sampling measurement")
    ap.add_argument("--no-projection", action="store_true", help="skip the projected-layer measurement")
    ap.add_argument("--page-size", type=int, default=0,
                    help="lay the KV caches out in pages of this many slots (0: contiguous regions)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU oracle sample budget")
    ap.add_argument("--only", default="",
                    help="comma-separated parts to run alone, without the headline (for profiler captures): "
                         + ", ".join(ONLY_PARTS))
    a = ap.parse_args()
    bad = [x for x in a.only.split(",") if x and x not in ONLY_PARTS]
    if bad:
        ap.error(f"--only: unknown part(s) {bad}")
    return a


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------- work counts
def prefill_flops(w, lo=0, hi=None) -> float:
    return 4.0 * w.head_dim * w.num_q_heads * w.attended_pairs(lo, hi)


def decode_bytes(w, lo=0, hi=None, entry_bytes=2) -> float:
    """Algorithmic HBM bytes of the decode requests [lo, hi): cache read
    (K and V of the c_b cached entries, entry_bytes each: 2 for bf16, 1 for
    E4M3), the new token's qkv row, the K/V append and the output row."""
    hi = w.batch if hi is None else hi
    D, Hq, Hkv, e = w.head_dim, w.num_q_heads, w.num_kv_heads, entry_bytes
    total = 0
    for c in w.cache_lens[lo:hi]:
        total += 2 * c * Hkv * D * e + w.qkv_width * 2 + 2 * Hkv * D * e + Hq * D * 2
    return float(total)


def source_sha(*names) -> str:
    """Hash of the kernel sources with // comments and blank lines removed, so
    that recorded counters stay tied to the code, not to its comments."""
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "causal_gqa_attention_qkv_gb300", "csrc", n)) as f:
            for line in f:
                code = line.split("//", 1)[0].rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:12]


class L2Flush:
    """Evicts the L2 between timed steps (outside the timed events): a 256 MiB
    buffer is written, then another 256 MiB buffer is read.  The step then
    starts with none of its inputs in L2, and the flush's own dirty lines
    have been written back by the read instead of by the step's first loads
    (a write alone leaves up to the whole L2 dirty, about 126 MB that an
    HBM-bound step would otherwise write back inside its timed region)."""

    def __init__(self, device, torch):
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=device)
        self.r = torch.ones(64 << 20, dtype=torch.float32, device=device)
        self.k = 0

    def __call__(self):
        self.k += 1
        self.w.fill_(self.k & 0xFF)
        self.r.sum()


def recorded_traffic(kernel: str, sha: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summaries, if
    they were taken on the current source (same sha); else None."""
    pat = re.compile(r"traffic_per_launch\s+" + re.escape(kernel) + r"\s+(\d+)\s+sha=(\w+)")
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    for fn in sorted(os.listdir(pdir)):
        if not fn.endswith((".md", ".txt")):
            continue
        with open(os.path.join(pdir, fn)) as f:
            for m in pat.finditer(f.read()):
                if m.group(2) == sha:
                    return int(m.group(1))
    return None


# ----------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append({"sm": float(parts[1]), "max": float(parts[2]),
                             "power": float(parts[3]) if parts[3] not in ("[N/A]", "") else None,
                             "hw_slowdown": parts[5] == "Active", "hw_thermal_slowdown": parts[6] == "Active",
                             "sw_thermal_slowdown": parts[7] == "Active", "sw_power_cap": parts[8] == "Active"})
            except ValueError:
                continue
        if not rows:
            return None
        reasons = sorted({k for r in rows for k in ("hw_slowdown", "hw_thermal_slowdown",
                                                    "sw_thermal_slowdown", "sw_power_cap") if r[k]})
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------- ranks
def max_over_ranks(values, device="cpu"):
    """Element-wise maximum of per-rank timings over all ranks (identity
    without an initialised process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(work_per_rank: float, world: int, ms_max: float) -> float:
    """Aggregate throughput: the units every rank processed / the slowest rank's time."""
    return work_per_rank * world / (ms_max * 1e-3)


# ----------------------------------------------------------------- our arm
def env_rank():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


class Timed:
    """Issues one step of a packed workload as append/attend launch groups,
    with CUDA events on the launching stream between them."""

    def __init__(self, ds, torch):
        from causal_gqa_attention_qkv_gb300 import attn
        self.ds, self.torch, self.attn = ds, torch, attn

    def launches_per_step(self) -> int:
        return self.ds.launches()

    def run(self, ev):
        """ev: list of 5 events: start, after prefill append, after prefill
        attention, before the decode call, after it.  An absent part records
        no events of its own (each record takes about 2 us of device time):
        its slots are set to the event before it, so that part times 0."""
        ds, attn = self.ds, self.attn
        n = ds.n_prefill_tokens
        ev[0].record()
        if ds.kv_prefill is not None:
            attn.prefill_prepare(ds.cfg, ds.qkv[:n], ds.q_norm_w, ds.k_norm_w, ds.cu_seqlens,
                                 ds.kv_prefill, ds.q_stage[:n], ds.workspace)
            ev[1].record()
            attn.prefill_attend(ds.cfg, ds.q_stage[:n], ds.cu_seqlens, ds.max_seqlen, ds.kv_prefill,
                                ds.out[:n], ds.workspace)
            ev[2].record()
        else:
            ev[1] = ev[2] = ev[0]
        if ds.kv_decode is not None:
            ev[3] = ev[2]
            # the new tokens' K/V are appended inside the split kernel (one launch, two with a merge)
            attn.decode(ds.cfg, ds.qkv[n:], ds.q_norm_w, ds.k_norm_w, ds.max_cache_len, ds.kv_decode,
                        ds.out[n:], ds.workspace)
            ev[4].record()
        else:
            ev[3] = ev[4] = ev[2]


def measure(w, steps, warmup, device, torch, dist_on, page_size=0, kv_dtype="bf16"):
    """Device-timed steps of workload w.  Returns per-part mean ms and more."""
    from causal_gqa_attention_qkv_gb300 import inputs as gen
    from causal_gqa_attention_qkv_gb300 import step

    host = gen.make_inputs(w, page_size=page_size, kv_dtype=kv_dtype)
    ds = step.upload(w, host, device=device)
    B_dec = w.batch - w.decode_from
    ds.decode_cu = torch.arange(B_dec + 1, dtype=torch.int32, device=device)
    ds.q_stage = torch.empty((max(ds.n_prefill_tokens, 1), w.num_q_heads, w.head_dim), dtype=torch.bfloat16,
                             device=device)
    t = Timed(ds, torch)
    flush = L2Flush(device, torch)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    for _ in range(warmup):
        flush()
        t.run([torch.cuda.Event(enable_timing=True) for _ in range(5)])
    torch.cuda.synchronize()
    if dist_on:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for k in range(steps):
        flush()
        t.run(evs[k])
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if dist_on:
        torch.distributed.barrier()
    st = ds.status()
    if st != 0:
        raise RuntimeError(f"device status {st} after the timed steps")
    parts = {"prefill_append": [], "prefill_attend": [], "decode_append": [], "decode_attend": [], "step": []}
    for e in evs:
        parts["prefill_append"].append(e[0].elapsed_time(e[1]))
        parts["prefill_attend"].append(e[1].elapsed_time(e[2]))
        parts["decode_append"].append(e[2].elapsed_time(e[3]))
        parts["decode_attend"].append(e[3].elapsed_time(e[4]))
        parts["step"].append(e[0].elapsed_time(e[4]))
    mean = {k: sum(v) / len(v) for k, v in parts.items()}
    return {"ms": mean, "wall_s": wall, "launches": t.launches_per_step() * steps, "ds": ds,
            "host": host}


def measure_e2e(w, ds, host, steps, warmup, device, torch):
    """The same prefill through the public API from pinned host buffers:
    step.HostPrefill copies the qkv rows in, runs prepare + attention and
    copies the output rows out, in token chunks pipelined over five streams
    (copies in, prepare, attention on two streams in turn, copies out).
    Every copy is inside the timed events; the per-chunk metadata (int32
    cu_seqlens and cached lengths) is copied in with the first chunk."""
    from causal_gqa_attention_qkv_gb300 import step
    N = w.num_tokens
    chunk = max(4096, -(-N // 8))
    qkv_h = host["qkv"].pin_memory()
    out_h = torch.empty(ds.out.shape, dtype=ds.out.dtype).pin_memory()
    q_stage = torch.empty((N, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device=device)
    hp = step.HostPrefill(ds.cfg, ds.q_norm_w, ds.k_norm_w, ds.kv_prefill, ds.workspace, ds.qkv, q_stage, ds.out,
                          chunk_tokens=chunk)
    plan = hp.plan(host["cu_seqlens"].tolist(), host["cache_lens"].tolist())
    h2d = qkv_h.numel() * 2 + plan.h2d_bytes
    d2h = out_h.numel() * 2
    times, launches = [], 0
    for k in range(warmup + steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n = hp.run(plan, qkv_h, out_h, e0, e1)
        e1.synchronize()
        if k >= warmup:
            times.append(e0.elapsed_time(e1))
            launches += n
    if ds.status() != 0 or hp.status() != 0:
        raise RuntimeError("device status set in the end-to-end prefill")
    return sum(times) / len(times), h2d, d2h, launches, len(plan.chunks)


def cpu_oracle_rate(w, budget_s: float, seed: int = 0, host=None):
    """The oracle as it stands on a bounded seeded sample of (token, head)
    rows of workload w, grown until one call takes about budget_s / 2.
    Returns (FLOPs of the sampled rows, seconds, sample description, threads,
    host inputs).  The seconds include the oracle's full K/V prologue."""
    import numpy as np
    import oracle
    from causal_gqa_attention_qkv_gb300 import inputs as gen

    host = gen.make_inputs(w) if host is None else host
    cfg = oracle.cfg_of(w)
    g = np.random.default_rng(seed)
    all_tok = w.num_tokens
    t0 = time.perf_counter()
    oracle.step(cfg, host, rows=np.zeros((0, 2), dtype=np.int32))  # the K/V prologue alone
    t_prologue = time.perf_counter() - t0
    count = 16
    while True:
        toks = g.integers(0, all_tok, size=count).astype(np.int32)
        heads = g.integers(0, w.num_q_heads, size=count).astype(np.int32)
        rows = np.stack([toks, heads], 1)
        t0 = time.perf_counter()
        oracle.step(cfg, host, rows=rows)
        dt = time.perf_counter() - t0
        if dt >= budget_s * 0.5 or count >= all_tok * w.num_q_heads:
            break
        count = int(min(count * max(2.0, budget_s / max(dt, 1e-3) * 0.8), all_tok * w.num_q_heads))
    cu = host["cu_seqlens"].numpy()
    cl = host["cache_lens"].numpy()
    b = np.searchsorted(cu, toks, side="right") - 1
    keys = cl[b] + (toks - cu[b]) + 1
    flops = 4.0 * w.head_dim * float(keys.sum())
    cpu_oracle_rate.t_prologue = t_prologue
    return flops, dt, f"{count} random (token, head) rows of {w.name}, with the full K/V prologue", \
        oracle.num_threads(), host


def cpu_oracle_decode_rate(w, budget_s: float, host=None):
    """The oracle on every head of the first nb decode requests of w (nb grown
    until one call takes about budget_s / 2).  Returns (algorithmic decode
    bytes of those requests, seconds, description, threads)."""
    import numpy as np
    import oracle
    from causal_gqa_attention_qkv_gb300 import inputs as gen

    host = gen.make_inputs(w) if host is None else host
    cfg = oracle.cfg_of(w)
    lo = w.decode_from
    nb = 1
    while True:
        reqs = np.arange(lo, lo + nb, dtype=np.int64)
        toks = host["cu_seqlens"].numpy()[reqs].astype(np.int32)
        rows = np.stack([np.repeat(toks, w.num_q_heads),
                         np.tile(np.arange(w.num_q_heads, dtype=np.int32), nb)], 1)
        t0 = time.perf_counter()
        oracle.step(cfg, host, rows=rows)
        dt = time.perf_counter() - t0
        if dt >= budget_s * 0.5 or nb >= w.batch - lo:
            break
        nb = int(min(w.batch - lo, max(nb * 2, nb * budget_s / max(dt, 1e-3) * 0.8)))
    return decode_bytes(w, lo, lo + nb), dt, f"all heads of {nb} decode requests of {w.name}, with the full " \
        "K/V prologue", oracle.num_threads()


def cpu_baseline_prefill(w, budget_s, host, flops_total):
    """cpu_baseline entry for a prefill workload: the oracle's TFLOP/s on a
    row sample, and the full-workload oracle time extrapolated from it."""
    f, dt, desc, cores, _ = cpu_oracle_rate(w, budget_s, host=host)
    rate = f / dt
    t_pro = min(cpu_oracle_rate.t_prologue, dt)
    # full time = the prologue once + the attention rows at the sample's rate
    full = t_pro + (dt - t_pro) * flops_total / f
    return {"value": round(rate / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": desc, "seconds": round(dt, 2), "prologue_s": round(t_pro, 2),
            "full_workload_s": round(full, 1), "full_workload_s_kind": "extrapolated"}


def cpu_baseline_decode(w, budget_s, host, bytes_total):
    b, dt, desc, cores = cpu_oracle_decode_rate(w, budget_s, host=host)
    rate = b / dt
    return {"value": round(rate / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": desc,
            "seconds": round(dt, 2), "full_workload_s": round(bytes_total / rate, 2),
            "full_workload_s_kind": "measured" if desc.startswith(f"all heads of {w.batch - w.decode_from} ")
            else "extrapolated"}


def measure_decode(wd, args, device, torch, dist_on, peaks, peak_kind, kv_dtype, entry_bytes,
                   traffic_kernel) -> dict:
    """The decode step (append + split-KV attention + combine) of workload wd
    over a cache of bf16 or E4M3 entries.  Bytes count the entries as stored."""
    md = measure(wd, args.steps, args.warmup, device, torch, dist_on, args.page_size, kv_dtype)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    dms, dcall = max_over_ranks([md["ms"]["step"], md["ms"]["decode_attend"]], device)
    nbytes = decode_bytes(wd, entry_bytes=entry_bytes)
    hbm = float(peaks["hbm_gbs"])
    return {
        "value": round(whole_job_rate(nbytes, world, dms) / 1e9, 1), "unit": "GB/s",
        "ms_per_step": round(dms, 4), "workload": wd.name, "kv_dtype": kv_dtype, "bytes_per_step": nbytes,
        "parts_ms": {"decode_split_and_merge": round(dcall, 4)},
        "roofline": {"bound": "hbm", "kernel": "decode split-KV (K/V append inside) + combine",
                     "bytes_per_launch": nbytes,
                     "achieved": round(nbytes / (dcall * 1e-3) / 1e9, 1), "peak": hbm,
                     "peak_kind": f"hbm_gbs ({peak_kind})", "unit": "GB/s",
                     "frac": round(nbytes / (dcall * 1e-3) / 1e9 / hbm, 4),
                     "frac_of_8tbs_nominal": round(nbytes / (dcall * 1e-3) / 8e12, 4),
                     "traffic": recorded_traffic(traffic_kernel, source_sha("decode.cu", "common.cuh"))},
        "gpu_launches": md["launches"],
        "host": md["host"],
    }


def cpu_wanted(args) -> bool:
    """The oracle baselines run on rank 0 of a single-process run only."""
    return env_rank()[0] == 0 and env_rank()[2] == 1 and not args.no_cpu


def measure_prefill(w, args, device, torch, dist_on, peaks, peak_kind, kv_dtype="bf16", e2e=False) -> dict:
    """The prefill step (prepare + attention) of workload w: TFLOP/s of the
    whole step, the attention kernel against the bf16 (f16 for an E4M3 cache)
    tensor peak, and optionally the same step end to end from host buffers."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    m = measure(w, args.steps, args.warmup, device, torch, dist_on, args.page_size, kv_dtype)
    step_ms, prep_ms, attend_ms = max_over_ranks([m["ms"]["step"], m["ms"]["prefill_append"],
                                                  m["ms"]["prefill_attend"]], device)
    flops = prefill_flops(w)
    achieved = flops / (attend_ms * 1e-3) / 1e12
    peak, peak_s = float(peaks["bf16_tflops"]), float(peaks.get("bf16_tflops_sustained", 0) or 0)
    qkv_bytes = 2.0 * w.num_tokens * w.qkv_width * 2  # prepare: read qkv, write K, V and prepared Q
    sha = source_sha("prefill_tc.cu", "tcgen05.cuh", "common.cuh")
    res = {
        "value": round(whole_job_rate(flops, world, step_ms) / 1e12, 3), "unit": "TFLOP/s",
        "ms_per_step": round(step_ms, 4), "workload": w.name, "kv_dtype": kv_dtype,
        "tokens": w.num_tokens, "attended_pairs": w.attended_pairs(), "flops_per_step": flops,
        "parts_ms": {"prologue": round(prep_ms, 4), "prefill_attention": round(attend_ms, 4)},
        "roofline": {"bound": "tensor",
                     "kernel": "prefill attention" + (" (E4M3 cache)" if kv_dtype == "e4m3" else ""),
                     "achieved": round(achieved, 3), "peak": peak, "peak_kind": f"bf16_tflops ({peak_kind})",
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "frac_of_sustained": round(achieved / peak_s, 4) if peak_s else None,
                     "traffic": recorded_traffic(f"prefill_attention_{w.name}" + ("_e4m3" if kv_dtype == "e4m3"
                                                                                  else ""), sha),
                     "flops_per_launch": flops},
        "prologue_roofline": {"bound": "hbm", "kernel": "kv_append_kernel (prefill prepare)",
                              "bytes_per_launch": qkv_bytes,
                              "achieved": round(qkv_bytes / (prep_ms * 1e-3) / 1e9, 1),
                              "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                              "frac": round(qkv_bytes / (prep_ms * 1e-3) / 1e9 / float(peaks["hbm_gbs"]), 4)},
        "gpu_launches": m["launches"],
    }
    if e2e:
        e2e_ms, h2d, d2h, launches, nchunks = measure_e2e(w, m["ds"], m["host"], max(3, args.steps // 2), 2,
                                                          device, torch)
        (e2e_ms,) = max_over_ranks([e2e_ms], device)
        res["e2e"] = {"value": round(flops * world / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                      "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                      "chunks": nchunks, "api": "step.HostPrefill (pinned host buffers, copies overlapped)"}
        res["gpu_launches"] += launches
    res["host"] = m["host"]
    del m
    return res


def measure_tiny(args, device, torch, dist_on) -> dict:
    """The tiny workload (12-token prompt, Hq 4 / Hkv 2 / D 64, then the
    decode step at position 12): microseconds per call through the public
    calls, launch-latency bound (5 warm-up calls, then the median of the
    timed ones, each bracketed by CUDA events); then both calls recorded
    into one CUDA graph and replayed, timed the same way."""
    from causal_gqa_attention_qkv_gb300 import inputs as gen
    from causal_gqa_attention_qkv_gb300 import step
    w = gen.tiny()
    host = gen.make_inputs(w)
    pre = step.upload(w, host, device=device)
    dw = gen.custom("tiny_decode", w.num_q_heads, w.num_kv_heads, w.head_dim, [1], [12], seed=0, decode_from=0)
    dhost = dict(host, qkv=gen.make_followup_decode_qkv(w), cu_seqlens=torch.tensor([0, 1], dtype=torch.int32),
                 cache_lens=torch.tensor([12], dtype=torch.int32))
    dec = step.upload(dw, dhost, device=device)
    res = {"workload": w.name, "unit": "us per call"}
    launches = 0
    for key, ds in (("prefill_us", pre), ("decode_us", dec)):
        for _ in range(max(5, args.warmup)):
            ds.run()
        torch.cuda.synchronize()
        if dist_on:
            torch.distributed.barrier()
        times = []
        for _ in range(args.steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            ds.run()
            e1.record()
            e1.synchronize()
            times.append(e0.elapsed_time(e1) * 1e3)
        (us,) = max_over_ranks([statistics.median(times)], device)
        res[key] = round(us, 2)
        launches += ds.launches() * args.steps
        if ds.status() != 0:
            raise RuntimeError("device status set on the tiny workload")
    # the same two calls recorded once into a CUDA graph and replayed: the
    # launch floor without the per-call host work
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pre.run()
        dec.run()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pre.run()
        dec.run()
    for _ in range(max(5, args.warmup)):
        g.replay()
    torch.cuda.synchronize()
    times = []
    for _ in range(args.steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        e1.synchronize()
        times.append(e0.elapsed_time(e1) * 1e3)
    (us,) = max_over_ranks([statistics.median(times)], device)
    res["graph_prefill_and_decode_us"] = round(us, 2)
    launches += (pre.launches() + dec.launches()) * args.steps
    if pre.status() != 0 or dec.status() != 0:
        raise RuntimeError("device status set on the tiny workload (graph replay)")
    res["gpu_launches"] = launches
    res["host"] = host
    res["decode_host"] = dhost
    return res


def measure_projection(w, args, device, torch, dist_on, peaks, peak_kind, hidden=2560) -> dict:
    """The attention layer with its projections (code walkthrough section
    3.3): the merged Q/K/V projection fused with the prologue, the prefill
    attention and the output projection, back to back on one stream, on
    workload w with a Qwen3-4B hidden size.  FLOPs: 2 N C (Hq + 2 Hkv) D for
    qkv_proj, 4 D Hq P for the attention, 2 N (Hq D) C for o_proj."""
    from causal_gqa_attention_qkv_gb300 import attn
    from causal_gqa_attention_qkv_gb300 import inputs as gen
    from causal_gqa_attention_qkv_gb300 import step
    host = gen.make_inputs(w, page_size=args.page_size)
    pr = gen.make_projection_inputs(w, hidden=hidden, seed=1)
    ds = step.upload(w, host, device=device)
    N = w.num_tokens
    hid, wq, wo = (pr[k].to(device) for k in ("hidden", "w_qkv", "w_o"))
    q = torch.empty((N, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device=device)
    att = torch.empty((N, w.num_q_heads * w.head_dim), dtype=torch.bfloat16, device=device)
    o = torch.empty((N, hidden), dtype=torch.bfloat16, device=device)
    kv, ws = ds.kv_prefill, ds.workspace
    flush = L2Flush(device, torch)

    def run(ev):
        ev[0].record()
        attn.qkv_proj_prepare(ds.cfg, hid, wq, ds.q_norm_w, ds.k_norm_w, ds.cu_seqlens, kv, q, ws)
        ev[1].record()
        attn.prefill_attend(ds.cfg, q, ds.cu_seqlens, ds.max_seqlen, kv, att, ws)
        ev[2].record()
        attn.o_proj(ds.cfg, att, wo, o, ws)
        ev[3].record()

    mk = lambda: [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for _ in range(args.warmup):
        flush()
        run(mk())
    torch.cuda.synchronize()
    if dist_on:
        torch.distributed.barrier()
    evs = [mk() for _ in range(args.steps)]
    for k in range(args.steps):
        flush()
        run(evs[k])
    torch.cuda.synchronize()
    if ds.status() != 0:
        raise RuntimeError("device status set in the projected step")
    mean = lambda i, j: sum(e[i].elapsed_time(e[j]) for e in evs) / len(evs)
    t_qkv, t_att, t_o, t_step = max_over_ranks([mean(0, 1), mean(1, 2), mean(2, 3), mean(0, 3)], device)
    f_qkv = 2.0 * N * hidden * w.qkv_width
    f_att = prefill_flops(w)
    f_o = 2.0 * N * w.num_q_heads * w.head_dim * hidden
    peak = float(peaks["bf16_tflops"])
    world = int(os.environ.get("WORLD_SIZE", "1"))
    tf = lambda f, ms: f / (ms * 1e-3) / 1e12
    return {
        "workload": f"{w.name}_hidden{hidden}", "value": round(whole_job_rate(f_qkv + f_att + f_o, world, t_step) / 1e12, 3),
        "unit": "TFLOP/s", "ms_per_step": round(t_step, 4),
        "flops": {"qkv_proj": f_qkv, "attention": f_att, "o_proj": f_o},
        "parts_ms": {"qkv_proj_prepare": round(t_qkv, 4), "prefill_attention": round(t_att, 4),
                     "o_proj": round(t_o, 4)},
        "roofline": {"bound": "tensor", "kernel": "proj_gemm_kernel (qkv projection + prologue epilogue)",
                     "achieved": round(tf(f_qkv, t_qkv), 3), "peak": peak,
                     "peak_kind": f"bf16_tflops ({peak_kind})", "unit": "TFLOP/s",
                     "frac": round(tf(f_qkv, t_qkv) / peak, 4)},
        "o_proj_roofline": {"bound": "tensor", "kernel": "proj_gemm_kernel (plain epilogue)",
                            "achieved": round(tf(f_o, t_o), 3), "peak": peak, "unit": "TFLOP/s",
                            "frac": round(tf(f_o, t_o) / peak, 4)},
        "gpu_launches": 3 * args.steps,
    }


def measure_sampling(args, device, torch, dist_on, peaks, peak_kind, B=64) -> dict:
    """Token sampling (temperature + top-k + top-p, no greedy rows) from fp32
    logits of B rows over the Qwen3 vocabulary: one kernel launch per step.
    Bytes: the logits and the per-row parameters read, the tokens written."""
    from causal_gqa_attention_qkv_gb300 import attn
    from causal_gqa_attention_qkv_gb300 import inputs as gen
    h = gen.make_sampling_inputs(B, gen.QWEN3_VOCAB, seed=6, greedy_share=0.0)
    d = {k: v.to(device) for k, v in h.items()}
    tokens = torch.empty(B, dtype=torch.int32, device=device)
    flush = L2Flush(device, torch)
    run = lambda: attn.sample_tokens(d["logits"], d["temperature"], d["top_k"], d["top_p"], d["uniform"], tokens)
    for _ in range(args.warmup):
        flush()
        run()
    torch.cuda.synchronize()
    if dist_on:
        torch.distributed.barrier()
    times = []
    for k in range(args.steps):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        run()
        e1.record()
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    (ms,) = max_over_ranks([sum(times) / len(times)], device)
    nbytes = B * gen.QWEN3_VOCAB * 4 + B * 4 * 4 + B * 4
    hbm = float(peaks["hbm_gbs"])
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": f"sample_b{B}_v{gen.QWEN3_VOCAB}_topk_topp_temperature", "ms_per_step": round(ms, 4),
            "rows_per_s": round(B / (ms * 1e-3), 1), "bytes_per_step": nbytes,
            "roofline": {"bound": "hbm", "kernel": "sample_kernel", "achieved": round(gbs, 1), "peak": hbm,
                         "peak_kind": f"hbm_gbs ({peak_kind})", "unit": "GB/s", "frac": round(gbs / hbm, 4)},
            "gpu_launches": args.steps}


def measure_mixed(wm, args, device, torch, dist_on, peaks, peak_kind) -> dict:
    """One serving step that mixes prefill chunks (on top of cached prefixes)
    with decode rows: the chunks' prepare + attention and the decode rows
    (append inside the split kernel) with their merge.  parts_ms and
    serial_ms_per_step time the parts one after the other on one stream;
    ms_per_step times the step as step.DeviceStep.run issues it, the decode
    rows on a side stream beside the chunks.  The roofline fraction adds the
    tensor-bound and the HBM-bound parts:
    (chunk FLOPs / bf16 peak + decode bytes / HBM peak) / step time, the
    bound of the parts run one after the other; the overlapped fraction
    takes the larger of the two instead, the bound of the parts side by
    side."""
    mm = measure(wm, args.steps, args.warmup, device, torch, dist_on, args.page_size)
    ms = mm["ms"]
    # the step as step.DeviceStep.run issues it: the decode rows on a side
    # stream beside the prefill chunks (the parts above run one after the other)
    ds, flush = mm["ds"], L2Flush(device, torch)
    for _ in range(args.warmup):
        flush()
        ds.run()
    torch.cuda.synchronize()
    times = []
    for _ in range(args.steps):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        ds.run()
        e1.record()
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    if ds.status() != 0:
        raise RuntimeError("device status set in the overlapped mixed step")
    step_ms, serial_ms, pp, pa, dd = max_over_ranks([sum(times) / len(times), ms["step"], ms["prefill_append"],
                                                     ms["prefill_attend"], ms["decode_attend"]], device)
    fl = prefill_flops(wm, 0, wm.decode_from)
    nb = decode_bytes(wm, wm.decode_from, wm.batch)
    peak_t, hbm = float(peaks["bf16_tflops"]) * 1e12, float(peaks["hbm_gbs"]) * 1e9
    ideal_s = fl / peak_t + nb / hbm
    return {
        "workload": wm.name, "ms_per_step": round(step_ms, 4), "serial_ms_per_step": round(serial_ms, 4),
        "chunk_flops": fl, "decode_bytes": nb,
        "roofline_frac": round(ideal_s / (step_ms * 1e-3), 4),
        # with the parts overlapped the bound is the larger of the two, not their sum
        "roofline_frac_overlapped": round(max(fl / peak_t, nb / hbm) / (step_ms * 1e-3), 4),
        "roofline_peaks": f"bf16_tflops and hbm_gbs ({peak_kind})",
        "parts_ms": {"chunk_prepare": round(pp, 4), "chunk_attention": round(pa, 4),
                     "decode_rows": round(dd, 4)},
        "chunk_attention_tflops": round(fl / (pa * 1e-3) / 1e12, 2),
        "decode_rows_gbs": round(nb / (dd * 1e-3) / 1e9, 1),
        "gpu_launches": mm["launches"] + ds.launches() * args.steps,
        "host": mm["host"],
    }


def run_only(args, device, torch, dist_on, peaks, peak_kind, rank):
    """The named parts alone, each with its own warm-up and timed steps, and
    no oracle: a short, fixed sequence of launches for profiler captures.
    Prints one JSON line with the parts' results."""
    from causal_gqa_attention_qkv_gb300 import inputs as gen
    parts = [x for x in args.only.split(",") if x]
    line = {"only": parts}
    for part in parts:
        if part in ("long_prefill", "prefill", "prefill_e4m3"):
            wl = gen.ALL[args.workload if part == "long_prefill" else args.prefill_workload]
            r = measure_prefill(wl, args, device, torch, dist_on, peaks, peak_kind,
                                kv_dtype="e4m3" if part == "prefill_e4m3" else "bf16")
        elif part in ("decode", "decode_e4m3"):
            f8 = part == "decode_e4m3"
            r = measure_decode(gen.ALL[args.decode_workload], args, device, torch, dist_on, peaks, peak_kind,
                               "e4m3" if f8 else "bf16", 1 if f8 else 2,
                               "decode_split_e4m3" if f8 else "decode_split")
        elif part == "mixed":
            r = measure_mixed(gen.ALL[args.mixed_workload], args, device, torch, dist_on, peaks, peak_kind)
        elif part == "projection":
            r = measure_projection(gen.ALL[args.prefill_workload], args, device, torch, dist_on, peaks, peak_kind)
        elif part == "tiny":
            r = measure_tiny(args, device, torch, dist_on)
        else:
            r = measure_sampling(args, device, torch, dist_on, peaks, peak_kind)
        for k in ("host", "ds", "decode_host"):
            r.pop(k, None)
        line[part] = r
    if dist_on:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_ours(args):
    import torch

    rank, local_rank, world = env_rank()
    dist_on = world > 1
    if dist_on:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    device = f"cuda:{local_rank}"
    from causal_gqa_attention_qkv_gb300 import attn, build
    from causal_gqa_attention_qkv_gb300 import inputs as gen
    if rank == 0 or not dist_on:
        build.build()
    if dist_on:
        torch.distributed.barrier()
    attn.load()
    peaks, peak_kind = load_peaks()
    cpu = cpu_wanted(args)
    pop = lambda d, *ks: [d.pop(k, None) for k in ks][0]
    if args.only:
        run_only(args, device, torch, dist_on, peaks, peak_kind, rank)
        return
    w = gen.ALL[args.workload]
    assert w.decode_from == w.batch, "the headline workload is a prefill workload"
    with ClockSampler(local_rank) as clk:
        head = measure_prefill(w, args, device, torch, dist_on, peaks, peak_kind, e2e=True)
    clocks = clk.summary()
    host = pop(head, "host")
    line = {
        "metric": METRIC, "value": head["value"], "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) qkv, norm weights 1+0.1N(0,1), no trained weights)",
        "config": {"workload": w.name, "global_batch": w.batch * world, "seq_len": max(w.new_lens),
                   "tokens": w.num_tokens, "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
                   "head_dim": w.head_dim, "attended_pairs": w.attended_pairs(),
                   "parallelism": f"replicas{world}",
                   "l2": "flushed before every timed step (256 MiB written, then 256 MiB read)",
                   "kv_layout": f"paged{args.page_size}" if args.page_size else "contiguous"},
        "parts_ms": head["parts_ms"], "roofline": head["roofline"],
        "prologue_roofline": head["prologue_roofline"],
        "gpu_launches": head["gpu_launches"], "e2e": head["e2e"], "clocks": clocks,
    }
    if cpu:
        line["cpu_baseline"] = cpu_baseline_prefill(w, args.cpu_seconds, host, head["flops_per_step"])
    del host
    # the Qwen3-4B-shaped prefill, over bf16 and over one-byte (E4M3) caches
    wp = gen.ALL[args.prefill_workload]
    for key, kvd in (("qwen3_4b_prefill", "bf16"), ("prefill_e4m3", "e4m3")):
        r = measure_prefill(wp, args, device, torch, dist_on, peaks, peak_kind, kv_dtype=kvd, e2e=kvd == "bf16")
        h = pop(r, "host")
        if cpu and kvd == "bf16":
            r["cpu_baseline"] = cpu_baseline_prefill(wp, args.cpu_seconds / 2, h, r["flops_per_step"])
        line[key] = r
        line["gpu_launches"] += r["gpu_launches"]
        del h
    if not args.no_decode:
        wd = gen.ALL[args.decode_workload]
        for key, kvd, eb, kname in (("decode", "bf16", 2, "decode_split"),
                                    ("decode_e4m3", "e4m3", 1, "decode_split_e4m3")):
            r = measure_decode(wd, args, device, torch, dist_on, peaks, peak_kind, kvd, eb, kname)
            h = pop(r, "host")
            if cpu and kvd == "bf16":
                r["cpu_baseline"] = cpu_baseline_decode(wd, args.cpu_seconds / 2, h, r["bytes_per_step"])
            line[key] = r
            line["gpu_launches"] += r["gpu_launches"]
    if not args.no_mixed:
        wm = gen.ALL[args.mixed_workload]
        r = measure_mixed(wm, args, device, torch, dist_on, peaks, peak_kind)
        h = pop(r, "host")
        if cpu:
            r["cpu_baseline"] = cpu_baseline_prefill(wm, args.cpu_seconds / 2, h, prefill_flops(wm))
            r["cpu_baseline"]["sample"] += " (chunk and decode rows alike; FLOPs over all attended pairs)"
        line["mixed"] = r
        line["gpu_launches"] += r["gpu_launches"]
    if not args.no_projection:
        line["projection"] = measure_projection(wp, args, device, torch, dist_on, peaks, peak_kind)
        line["gpu_launches"] += line["projection"]["gpu_launches"]
    r = measure_tiny(args, device, torch, dist_on)
    h, dh = pop(r, "host"), pop(r, "decode_host")
    if cpu:
        import oracle
        wt = gen.tiny()
        cfg = oracle.cfg_of(wt)
        t0 = time.perf_counter()
        reps = 0
        while time.perf_counter() - t0 < 0.5:
            oracle.step(cfg, h)
            oracle.step(cfg, dh)
            reps += 1
        per = (time.perf_counter() - t0) / reps
        r["cpu_baseline"] = {"value": round(per * 1e6, 1), "unit": "us per prefill + decode", "cores":
                             oracle.num_threads(), "kind": "oracle", "sample": f"the whole workload, {reps} times",
                             "full_workload_s_kind": "measured"}
    line["tiny"] = r
    line["gpu_launches"] += r["gpu_launches"]
    if not args.no_sampling:
        line["sampling"] = measure_sampling(args, device, torch, dist_on, peaks, peak_kind)
        line["gpu_launches"] += line["sampling"]["gpu_launches"]
    if dist_on:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_reference(args):
    rank, _, world = env_rank()
    if rank != 0:
        return
    from causal_gqa_attention_qkv_gb300 import inputs as gen
    w = gen.ALL[args.workload]
    per_step = max(1.0, min(6.0, 150.0 / max(1, args.steps + args.warmup)))
    host = gen.make_inputs(w)
    rates = []
    desc = cores = None
    for k in range(args.warmup + args.steps):
        flops, dt, desc, cores, _ = cpu_oracle_rate(w, per_step, seed=k, host=host)
        if k >= args.warmup:
            rates.append((flops, dt))
    tot_f = sum(f for f, _ in rates)
    tot_t = sum(t for _, t in rates)
    value = tot_f / tot_t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot_t / len(rates) * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": w.name, "global_batch": w.batch, "seq_len": max(w.new_lens),
                   "tokens": w.num_tokens, "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
                   "head_dim": w.head_dim, "attended_pairs": w.attended_pairs(),
                   "parallelism": "host cores (OpenMP)"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": desc + " per step",
                         "full_workload_s": round(cpu_oracle_rate.t_prologue + (tot_t / len(rates) -
                                                   cpu_oracle_rate.t_prologue) * prefill_flops(w) /
                                                  (tot_f / len(rates)), 1),
                         "full_workload_s_kind": "extrapolated"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
