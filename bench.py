"""Throughput of the batched multi-session decode step on GB300.

Workload (default): the Llama-3-8B-shaped dense model with random Q8_0 weights
(32 layers, hidden 4096, 32/8 heads of 128, FFN 14336, vocab 128256), B = 8
sessions, each slot pre-filled with 1238 random fp16 positions; every step
decodes one token per session at positions 1238 .. 1365 (cycling), so the
attended lengths stay within the 128-step decode window of the workload.

Prints ONE JSON line (rank 0): aggregate decode tok/s (`value`, inputs resident
on the device, steps issued back to back), achieved HBM GB/s, an end-to-end
number through the public API with a host round trip every step (`e2e`), the
dominant kernel's roofline, the B = 1..16 sweep, the CPU oracle's baseline and
the SM clocks seen during the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--batch B] [--no-sweep]
  python bench.py --impl reference ...   (the CPU oracle on the same workload)
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

PREFILL = synth.DENSE_8B_CASE["prefill"]
CAPACITY = synth.DENSE_8B_CASE["capacity"]
WINDOW = synth.DENSE_8B_CASE["steps"]  # positions PREFILL .. PREFILL+WINDOW-1
METRIC = "aggregate decode tok/s (8B-shaped Q8_0, B sessions, 1 GB300)"
FALLBACK_HBM_GBS = 6800.0


def kv_bytes_per_pos(s, kv_q8=False):
    """K and V bytes of one position over all layers and KV heads: fp16 rows, or
    Q8_0 rows (a quant byte per value and an fp16 scale per 32 values)."""
    row = s.head_dim + s.head_dim // 32 * 2 if kv_q8 else s.head_dim * 2
    return 2 * s.n_layers * s.n_kv_heads * row


def step_bytes(s, positions, kv_q8=False):
    """Algorithmic HBM bytes of one step: every weight once, the embedding rows,
    the KV rows attended (incl. the new one) and the new rows written."""
    B = len(positions)
    kvb = kv_bytes_per_pos(s, kv_q8)
    return (s.weight_bytes() + B * (s.hidden // 32) * 34 + sum(int(p) + 1 for p in positions) * kvb
            + B * kvb)


def kernels_per_step(s, with_argmax=True):
    # embed; per layer qkv, attention split, combine, o-proj, norm, gate|up, down, norm; lm_head; argmax
    # (the most a step launches; bench.py reports the count the library's profile saw)
    return 1 + s.n_layers * 8 + 1 + (1 if with_argmax else 0)


def max_over_ranks(value: float, world: int, device) -> float:
    """The largest of the ranks' values, returned on every rank (the value itself for one rank)."""
    if world <= 1:
        return value
    import torch
    t = torch.tensor([value], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_tok_s(batch: int, steps: int, world: int, seconds: float) -> float:
    """Tokens of all ranks (each rank decodes `batch` sessions for `steps` steps) over the slowest rank's time."""
    return batch * steps * world / seconds


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        for k in ("hbm_gbs", "hbm_GBps", "hbm_copy_gbs"):
            if k in d:
                return float(d[k]), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.25)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in self.rows:
            try:
                sm.append(float(r[0]))
                mx.append(float(r[1]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def sources_digest(paths):
    """First 16 hex digits of the sha256 of the listed files' bytes, concatenated in order."""
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_for(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel's sources are unchanged."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d[kernel]
        return e["dram_bytes_per_launch"] if sources_digest(e["sources"]) == e["sources_sha256_16"] else None
    except (OSError, ValueError, KeyError):
        return None


# --------------------------------------------------------------------------- ours
def run_kd(args, rank, world):
    import torch

    import session_decode_step_gb300 as kd
    from session_decode_step_gb300 import build as kbuild

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    kbuild.build()
    shape = synth.LLAMA3_8B
    B = args.batch
    max_b = 16 if args.sweep else B
    w = synth.model_weights(shape, seed=0)
    m = kd.kd_model_load(kd.make_config(shape, max_sessions=max_b, max_ctx=CAPACITY), w)
    ids = []
    for i in range(max_b):
        k, v = synth.kv_prefill(shape, 0, i, PREFILL)
        sid = kd.kd_session_bind(m)
        kd.kd_session_load_kv(m, sid, k, v, PREFILL)
        ids.append(sid)
        del k, v
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    tok = synth.tokens(0, "bench", max_b, shape.vocab)
    am = torch.empty(max_b, dtype=torch.int32, device=dev)

    def pos_at(i, b):
        return np.full(b, PREFILL + (i % WINDOW), np.int32)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    def timed(b, steps, warmup):
        for i in range(warmup):
            kd.kd_decode_step(m, ids[:b], tok[:b], pos_at(i, b), None, am[:b], stream)
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        byts = 0
        e0.record(stream)
        for i in range(warmup, warmup + steps):
            p = pos_at(i, b)
            kd.kd_decode_step(m, ids[:b], tok[:b], p, None, am[:b], stream)
            byts += step_bytes(shape, p)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
        return ms, byts

    gpu_index = local
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        try:
            gpu_index = int(vis.split(",")[local])
        except ValueError:
            pass
    with ClockSampler(gpu_index) as clk:
        ms, byts = timed(B, args.steps, args.warmup)
    status = kd.kd_device_status(m)
    tok_s = whole_job_tok_s(B, args.steps, world, ms / 1e3)
    gbs = byts / (ms / 1e3) / 1e9

    # ---- end to end through the public API: host tokens in, host argmax out, every step.
    # The loop does what a serving loop would: the step's host inputs (sessions,
    # tokens, positions) are host arrays, the argmax comes back into pinned host
    # memory, and its values are the next step's tokens (two pinned buffers swap).
    e2e_steps = min(args.steps, 128)
    ids_b = np.ascontiguousarray(ids[:B], dtype=np.int32)
    pos_tab = [pos_at(i, B) for i in range(max(args.warmup, e2e_steps))]
    am_b = am[:B]
    bufs = [torch.tensor(tok[:B], dtype=torch.int32).pin_memory(), torch.empty(B, dtype=torch.int32).pin_memory()]
    views = [b.numpy() for b in bufs]
    for i in range(args.warmup):
        kd.kd_decode_step(m, ids_b, views[0], pos_tab[i], None, am_b, stream)
        bufs[1].copy_(am_b, non_blocking=True)
        torch.cuda.synchronize()
    bufs[0].copy_(torch.tensor(tok[:B], dtype=torch.int32))
    barrier()
    t0 = time.perf_counter()
    cur = 0
    for i in range(e2e_steps):
        kd.kd_decode_step(m, ids_b, views[cur], pos_tab[i], None, am_b, stream)
        bufs[cur ^ 1].copy_(am_b, non_blocking=True)
        stream.synchronize()
        cur ^= 1  # greedy feedback through the host: this step's argmax is the next step's tokens
    e2e_s = max_over_ranks(time.perf_counter() - t0, world, dev)
    e2e = {"value": round(whole_job_tok_s(B, e2e_steps, world, e2e_s), 2), "unit": "tok/s",
           "h2d_bytes_per_step": 3 * 16 * 4, "d2h_bytes_per_step": B * 4, "steps": e2e_steps}

    # ---- per-kernel device times (events around every launch) for the roofline
    kd.kd_profile_enable(m, True)
    kd.kd_profile_read(m)
    n_prof = 8
    for i in range(n_prof):
        kd.kd_decode_step(m, ids[:B], tok[:B], pos_at(i, B), None, am[:B], stream)
    prof = kd.kd_profile_read(m)
    kd.kd_profile_enable(m, False)
    peak, peak_kind = read_peaks()
    wb = synth.Q8_BLOCK_BYTES / synth.Q8_BLOCK
    H, F = shape.hidden, shape.ffn
    per_launch_bytes = {
        "gate_up": 2 * F * H * wb + B * H * 2 + B * F * 2,
        "down": H * F * wb + B * F * 2 + 2 * B * H * 4,
        "qkv": (shape.q_dim + 2 * shape.kv_dim) * H * wb + B * H * 2 + B * shape.q_dim * 4 + 2 * B * shape.kv_dim * 2,
        "wo": H * shape.q_dim * wb + B * shape.q_dim * 2 + 2 * B * H * 4,
        "lm_head": shape.vocab * H * wb + B * H * 2 + B * shape.vocab * 4,
        "attn_split": (sum(PREFILL + (i % WINDOW) + 1 for i in range(n_prof)) / n_prof) * B
        * shape.n_kv_heads * shape.head_dim * 2 * 2,
    }
    dominant = max(prof, key=lambda k: prof[k][1])
    n_l, t_ms = prof[dominant]
    avg_s = t_ms / max(n_l, 1) / 1e3
    alg = per_launch_bytes.get(dominant)
    roofline = None
    if alg is not None and avg_s > 0:
        ach = alg / avg_s / 1e9
        roofline = {"bound": "hbm", "kernel": dominant, "achieved": round(ach, 1), "peak": peak,
                    "peak_source": peak_kind, "unit": "GB/s", "frac": round(ach / peak, 4),
                    "traffic": traffic_for(dominant), "alg_bytes_per_launch": int(alg),
                    "avg_launch_us": round(avg_s * 1e6, 2)}
    launches_per_step = sum(v[0] for v in prof.values()) / n_prof
    kernel_share = {k: {"launches": v[0], "ms": round(v[1], 3),
                        "share": round(v[1] / max(1e-9, sum(x[1] for x in prof.values())), 4)}
                    for k, v in prof.items()}

    # ---- B = 1 .. 16 sweep
    sweep = {}
    if args.sweep:
        for b in (1, 2, 4, 8, 16):
            sm, sb = timed(b, max(16, min(args.steps, 128)), args.warmup)
            n = max(16, min(args.steps, 128))
            sweep[str(b)] = {"tok_s": round(whole_job_tok_s(b, n, world, sm / 1e3), 1),
                             "hbm_gbs": round(sb / (sm / 1e3) / 1e9, 1),
                             "frac_of_peak": round(sb / (sm / 1e3) / 1e9 / peak, 4)}
    kd.kd_model_free(m)

    workloads = None
    if rank == 0 and args.workloads:
        workloads = other_workloads(args.steps, args.warmup, w if synth.LONG_CTX_8B_CASE["seed"] == 0 else None)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(shape, w, B)
    return dict(value=tok_s, ms=ms, gbs=gbs, e2e=e2e, roofline=roofline, sweep=sweep, cpu=cpu, workloads=workloads,
                clocks=clk.summary(), peak=peak, peak_kind=peak_kind, status=status, shares=kernel_share,
                launches_per_step=launches_per_step)


def cpu_baseline(shape, w, B):
    """The CPU oracle as it stands, one decode step of the B sessions (bounded sample)."""
    import oracle
    om = oracle.OracleModel(shape, w)
    cap = PREFILL + 1
    caches = [om.new_cache(cap, *synth.kv_prefill(shape, 0, i, PREFILL)) for i in range(B)]
    tok = synth.tokens(0, "bench", B, shape.vocab)
    t0 = time.perf_counter()
    om.step(tok, [PREFILL] * B, caches, cap)
    dt = time.perf_counter() - t0
    return {"value": round(B / dt, 4), "unit": "tok/s", "cores": len(os.sched_getaffinity(0)),
            "kind": "oracle",
            "sample": f"1 decode step of {B} sessions at position {PREFILL} (8B-shaped Q8_0, fp64 C oracle, "
                      f"OpenMP over rows), {dt:.1f} s"}


# --------------------------------------------------------------- op-level modes
def time_mmvq(R, K, m, steps, warmup):
    """Isolated Q8_0 mmvq (R x K weights, m fp16 activation rows ~N(0,1)).
    Distinct weight copies totalling more than 4x L2 are rotated, so every launch
    streams its weights from HBM."""
    import torch

    import session_decode_step_gb300 as kd
    wbytes = R * K * 34 // 32
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    copies = max(2, -(-4 * l2 // wbytes))
    base = synth.q8_0_matrix(0, f"op-{R}x{K}", R, K)
    hs = []
    for c in range(copies):  # distinct bytes per copy: rotate the quants, keep the scales
        w = base.copy()
        w[:, :, 2:] = np.roll(base[:, :, 2:], c, axis=2)
        hs.append(kd.kd_q8_matrix_create(w))
    x = torch.from_numpy(synth.activations_fp16(0, "op-x", m, K).view(np.int16)).cuda()
    y = torch.empty(m, R, device="cuda", dtype=torch.float32)
    st = torch.cuda.current_stream()
    for i in range(max(3, warmup)):
        kd.kd_mmvq(hs[i % copies], x, m, y, st)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for i in range(steps):
        kd.kd_mmvq(hs[i % copies], x, m, y, st)
    e1.record(st)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / steps
    alg = wbytes + m * K * 2 + m * R * 4
    peak, kind = read_peaks()
    status = max(kd.kd_q8_matrix_status(h) for h in hs)
    for h in hs:
        kd.kd_q8_matrix_free(h)
    return {"rows": R, "cols": K, "m": m, "copies": copies, "launches": steps,
            "avg_us": round(us, 3), "alg_bytes": alg, "gbs": round(alg / us / 1e3, 1), "peak": peak,
            "peak_source": kind, "frac": round(alg / us / 1e3 / peak, 4), "device_status": status}


def run_op_mmvq(args):
    import torch

    from session_decode_step_gb300 import build as kbuild
    kbuild.build()
    torch.cuda.set_device(0)
    return dict(op="mmvq", **time_mmvq(args.rows, args.cols, args.m, args.steps, args.warmup))


def time_attn(B, cap, steps, warmup, kv_q8=False):
    """Isolated KV append + ragged split-K flash-decode: 32/8 heads of 128, B sessions with
    attended lengths uniform in [1, cap] (seeded), KV ~N(0,1) in fp16 (or, kv_q8, those
    values quantised to Q8_0)."""
    import torch

    import session_decode_step_gb300 as kd
    c = synth.RAGGED_ATTN_CASE
    nh, nkv, hd = c["n_heads"], c["n_kv_heads"], c["head_dim"]
    lens = synth.ragged_lengths(0, "attn-config", B, 1, cap)
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    if kv_q8:
        planes = []
        for _ in range(2):
            x = torch.randn(B, nkv, cap, hd, device="cuda", generator=g)
            qs = torch.empty(B, nkv, cap, hd, dtype=torch.uint8, device="cuda")
            sc = torch.empty(B, nkv, cap, hd // 32, dtype=torch.int16, device="cuda")
            kd.kd_kv_q8_quantize(x, qs, sc)
            planes += [qs, sc]
            del x
        kc = vc = None
    else:
        kc = torch.randn(B, nkv, cap, hd, device="cuda", generator=g).to(torch.float16)
        vc = torch.randn(B, nkv, cap, hd, device="cuda", generator=g).to(torch.float16)
    q = torch.randn(B, nh, hd, device="cuda", generator=g)
    kn = torch.randn(B, nkv, hd, device="cuda", generator=g)
    vn = torch.randn(B, nkv, hd, device="cuda", generator=g)
    out = torch.empty(B, nh * hd, dtype=torch.float16, device="cuda")
    ws = torch.empty(kd.kd_attn_workspace_bytes(B, nh, hd, cap), dtype=torch.uint8, device="cuda")
    slots = np.arange(B, dtype=np.int32)
    pos = (lens - 1).astype(np.int32)
    st = torch.cuda.current_stream()

    def call():
        if kv_q8:
            kd.kd_attn_append_decode_q8(q, kn, vn, *planes, slots, pos, nh, nkv, B, cap, out, ws, st)
        else:
            kd.kd_attn_append_decode(q, kn, vn, kc, vc, slots, pos, nh, nkv, hd, B, cap, out, ws, st)
    for _ in range(max(3, warmup)):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(steps):
        call()
    e1.record(st)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / steps
    row = hd + hd // 32 * 2 if kv_q8 else hd * 2  # K or V bytes of one head row
    alg = int(lens.sum()) * nkv * row * 2 + B * nkv * row * 2
    peak, kind = read_peaks()
    status = kd.kd_attn_device_status(ws, st)
    return {"B": B, "cap": cap, "kv": "q8_0" if kv_q8 else "fp16", "sum_t_kv": int(lens.sum()), "launches": steps,
            "avg_us": round(us, 3), "alg_bytes": alg, "gbs": round(alg / us / 1e3, 1), "peak": peak,
            "peak_source": kind, "frac": round(alg / us / 1e3 / peak, 4), "device_status": status,
            "note": "per call: host-staged descriptor copy, append, split kernel, combine"}


def run_op_attn(args):
    import torch

    from session_decode_step_gb300 import build as kbuild
    kbuild.build()
    torch.cuda.set_device(0)
    return dict(op="attn_append_decode", **time_attn(args.m, args.cap, args.steps, args.warmup, args.kv_q8))


def time_long(steps, warmup, w=None, kv_q8=False):
    """The long-context multi-tenant workload: 8 sessions in 32768-position slots, pre-filled to
    25704 + 1000 i (i = 0..7) fp16 positions, each step at its own position (64 positions cycling);
    kv_q8: the cache held as Q8_0 (KD_FLAG_KV_Q8_0)."""
    import torch

    import session_decode_step_gb300 as kd
    c = synth.LONG_CTX_8B_CASE
    shape, S, cap, win = c["shape"], c["sessions"], c["capacity"], c["steps"]
    lens = [c["prefill_base"] + c["prefill_stagger"] * i for i in range(S)]
    if w is None:
        w = synth.model_weights(shape, seed=c["seed"])
    m = kd.kd_model_load(kd.make_config(shape, max_sessions=S, max_ctx=cap,
                                        flags=kd.KD_FLAG_KV_Q8_0 if kv_q8 else 0), w)
    ids = []
    for i, n in enumerate(lens):
        k, v = synth.kv_prefill(shape, c["seed"], 1000 + i, n)
        sid = kd.kd_session_bind(m)
        kd.kd_session_load_kv(m, sid, k, v, n)
        torch.cuda.synchronize()
        ids.append(sid)
        del k, v
    tok = synth.tokens(c["seed"], "bench-long", S, shape.vocab)
    am = torch.empty(S, dtype=torch.int32, device="cuda")
    st = torch.cuda.current_stream()

    def pos(i):
        return np.array([n + (i % win) for n in lens], np.int32)

    for i in range(max(3, warmup)):
        kd.kd_decode_step(m, ids, tok, pos(i), None, am, st)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    byts = 0
    e0.record(st)
    for i in range(steps):
        p = pos(i)
        kd.kd_decode_step(m, ids, tok, p, None, am, st)
        byts += step_bytes(shape, p, kv_q8)
    e1.record(st)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    peak, kind = read_peaks()
    status = kd.kd_device_status(m)
    kd.kd_model_free(m)
    return {"B": S, "capacity": cap, "kv": "q8_0" if kv_q8 else "fp16", "positions": f"{lens[0]}..{lens[-1] + win - 1}",
            "steps": steps, "ms_per_step": round(ms, 4), "tok_s": round(S / (ms / 1e3), 1),
            "alg_bytes_per_step": int(byts / steps), "gbs": round(byts / steps / (ms / 1e3) / 1e9, 1),
            "peak": peak, "peak_source": kind, "frac": round(byts / steps / (ms / 1e3) / 1e9 / peak, 4),
            "device_status": status}


def run_op_long(args):
    import torch

    from session_decode_step_gb300 import build as kbuild
    kbuild.build()
    torch.cuda.set_device(0)
    return dict(op="long_context_step", **time_long(args.steps, args.warmup, kv_q8=args.kv_q8))


def run_op_step(args):
    """The 8B-shaped step (hidden 4096, 32/8 heads of 128, FFN 14336, vocab 128256) with
    `--layers` decoder layers, B = `--batch` sessions pre-filled to 1238 positions: the
    same kernels and launch train at a depth whose device footprint (about 1.6 GB at 2
    layers) suits profiler captures of single launches."""
    import dataclasses

    import torch

    import session_decode_step_gb300 as kd
    from session_decode_step_gb300 import build as kbuild
    kbuild.build()
    torch.cuda.set_device(0)
    shape = dataclasses.replace(synth.LLAMA3_8B, name=f"llama3-8b-shaped-{args.layers}L", n_layers=args.layers)
    B = args.batch
    w = synth.model_weights(shape, seed=0)
    m = kd.kd_model_load(kd.make_config(shape, max_sessions=B, max_ctx=CAPACITY), w)
    ids = []
    for i in range(B):
        k, v = synth.kv_prefill(shape, 0, i, PREFILL)
        sid = kd.kd_session_bind(m)
        kd.kd_session_load_kv(m, sid, k, v, PREFILL)
        ids.append(sid)
    tok = synth.tokens(0, "bench", B, shape.vocab)
    am = torch.empty(B, dtype=torch.int32, device="cuda")
    st = torch.cuda.current_stream()
    for i in range(args.warmup):
        kd.kd_decode_step(m, ids, tok, np.full(B, PREFILL + i, np.int32), None, am, st)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for i in range(args.steps):
        kd.kd_decode_step(m, ids, tok, np.full(B, PREFILL + (args.warmup + i) % WINDOW, np.int32), None, am, st)
    e1.record(st)
    torch.cuda.synchronize()
    status = kd.kd_device_status(m)
    kd.kd_model_free(m)
    return {"op": "step", "layers": args.layers, "B": B, "steps": args.steps,
            "ms_per_step": round(e0.elapsed_time(e1) / args.steps, 4), "device_status": status}


def run_op_timeline(args):
    """Where the graph-replayed step's time goes: per-CTA global-timer stamps of every
    launch (kd_profile_timeline) of the 8B-shaped step at B = --batch (1238 positions),
    or with --long the long-context case (8 sessions at 25704 + 1000 i positions, KV in
    fp16 or with --kv-q8 in Q8_0), summarised per kernel class over the middle layers
    (medians): `run` = the first CTA's dependency release to the last CTA's end, `gap`
    = that end to the next kernel's first release, `early` = the first CTA's entry to
    the release."""
    import torch

    import session_decode_step_gb300 as kd
    from session_decode_step_gb300 import build as kbuild
    kbuild.build()
    torch.cuda.set_device(0)
    shape = synth.LLAMA3_8B
    if args.long:
        c = synth.LONG_CTX_8B_CASE
        cap, win = c["capacity"], c["steps"]
        lens = [c["prefill_base"] + c["prefill_stagger"] * i for i in range(c["sessions"])]
    else:
        cap, win = CAPACITY, WINDOW
        lens = [PREFILL] * args.batch
    B = len(lens)
    w = synth.model_weights(shape, seed=0)
    flags = kd.KD_FLAG_KV_Q8_0 if args.kv_q8 else 0
    m = kd.kd_model_load(kd.make_config(shape, max_sessions=B, max_ctx=cap, flags=flags), w)
    ids = []
    for i in range(B):
        k, v = synth.kv_prefill(shape, 0, i, lens[i])
        sid = kd.kd_session_bind(m)
        kd.kd_session_load_kv(m, sid, k, v, lens[i])
        torch.cuda.synchronize()
        ids.append(sid)
        del k, v
    tok = synth.tokens(0, "bench", B, shape.vocab)
    am = torch.empty(B, dtype=torch.int32, device="cuda")
    st = torch.cuda.current_stream()
    nmax = 1 + shape.n_layers * 8 + 3
    buf = torch.zeros(nmax, kd.KD_TIMELINE_CTAS, 4, dtype=torch.int64, device="cuda")
    classes = kd.kd_profile_timeline(m, buf, nmax)
    n_launch = sum(c is not None for c in classes)
    # embed, the layers (layer 0's attention norm is formed by the embedding
    # kernel), the output norm, lm_head (and argmax, unless lm_head made the pick)
    qkv_at = [j for j in range(n_launch) if classes[j] == "qkv"]
    head_at = classes.index("lm_head")
    tail = [(0, "embed"), (head_at - 1, "rmsnorm_out"), (head_at, "lm_head")]
    if head_at + 1 < n_launch:
        tail.append((head_at + 1, "argmax"))
    stats, steps_ns = {}, []
    for i in range(max(3, args.warmup) + args.steps):
        buf.zero_()
        kd.kd_decode_step(m, ids, tok, np.array(lens, np.int32) + i % win, None, am, st)
        torch.cuda.synchronize()
        if i < max(3, args.warmup):
            continue
        t = buf.cpu().numpy()
        rows = []
        for j in range(n_launch):
            r = t[j][t[j][:, 0] > 0]
            rows.append((int(r[:, 0].min()), int(r[:, 1].min()), int(r[:, 2].max()), len(r)))
        steps_ns.append(rows[-1][2] - rows[0][0])
        for j in range(qkv_at[2] - 1, qkv_at[shape.n_layers - 2] - 1):  # layers 2 .. L - 3, from their norm
            name = classes[j]
            if name == "rmsnorm":
                name += "_ffn" if classes[j + 1] == "gate_up" else "_attn"
            d = stats.setdefault(name, {"run": [], "gap": [], "early": [], "ctas": rows[j][3]})
            d["run"].append((rows[j][2] - rows[j][1]) / 1e3)
            d["gap"].append((rows[j + 1][1] - rows[j][2]) / 1e3)
            d["early"].append((rows[j][1] - rows[j][0]) / 1e3)
        for j, name in tail:
            d = stats.setdefault(name, {"run": [], "gap": [], "early": [], "ctas": rows[j][3]})
            d["run"].append((rows[j][2] - rows[j][1]) / 1e3)
            d["gap"].append((rows[j + 1][1] - rows[j][2]) / 1e3 if j + 1 < n_launch else 0.0)
            d["early"].append((rows[j][1] - rows[j][0]) / 1e3)
    kd.kd_profile_timeline(m, None)
    kd.kd_model_free(m)
    summ = {k: {"run_us": round(statistics.median(v["run"]), 2), "gap_us": round(statistics.median(v["gap"]), 2),
                "early_us": round(statistics.median(v["early"]), 2), "ctas": v["ctas"]} for k, v in stats.items()}
    layer_us = sum(v["run_us"] + v["gap_us"] for k, v in summ.items()
                   if k not in ("embed", "rmsnorm_out", "lm_head", "argmax"))
    return {"op": "timeline", "B": B, "positions": f"{lens[0]}..{lens[-1] + win - 1}", "kv": "q8_0" if args.kv_q8 else "fp16",
            "steps": args.steps, "step_us": round(statistics.median(steps_ns) / 1e3, 1),
            "launches_per_step": n_launch, "layer_us": round(layer_us, 2), "classes": summ}


def other_workloads(steps, warmup, w):
    """The workloads other than the headline one, measured in the same run: the
    long-context step, the isolated mmvq at every m, the isolated ragged attention."""
    c2, c3 = synth.MMVQ_CASE, synth.RAGGED_ATTN_CASE
    nl = max(16, min(steps, synth.LONG_CTX_8B_CASE["steps"]))
    out = {"long_context": time_long(nl, warmup, w), "long_context_kv_q8": time_long(nl, warmup, w, kv_q8=True)}
    out["isolated_mmvq"] = [time_mmvq(R, K, m, max(50, min(steps, 200)), warmup)
                            for R, K in c2["matrices"] for m in c2["rows_m"]]
    out["isolated_attention"] = time_attn(c3["sessions"], c3["max_ctx"], max(50, min(steps, 200)), warmup)
    out["isolated_attention_kv_q8"] = time_attn(c3["sessions"], c3["max_ctx"], max(50, min(steps, 200)), warmup,
                                                kv_q8=True)
    return out


# ------------------------------------------------------------------ reference arm
def run_reference(args):
    """The oracle timed as it stands on the host cores, one layer of one session per step."""
    import oracle
    shape = synth.LLAMA3_8B
    B = args.batch
    w = synth.model_weights(shape, seed=0)
    om = oracle.OracleModel(shape, w)
    cap = PREFILL + WINDOW
    caches = [om.new_cache(cap, *synth.kv_prefill(shape, 0, i, PREFILL)) for i in range(B)]
    x = [np.zeros(shape.hidden) for _ in range(B)]
    for b in range(B):  # embedding rows as the start of each session's residual stream
        x[b][:] = oracle.q8_0_dequant_row(w["tok_embd"][int(synth.tokens(0, "bench", B, shape.vocab)[b])],
                                          shape.hidden)

    def one(i):
        b, l = i % B, (i // B) % shape.n_layers
        om.layer_step(l, PREFILL + (i // (B * shape.n_layers)) % WINDOW, caches[b], cap, x[b])

    for i in range(args.warmup):
        one(i)
    t0 = time.perf_counter()
    for i in range(args.warmup, args.warmup + args.steps):
        one(i)
    dt = time.perf_counter() - t0
    per_layer = dt / args.steps
    tok_s = 1.0 / (per_layer * shape.n_layers)
    cores = len(os.sched_getaffinity(0))
    sample = (f"each step = one decoder layer of one session (1/{shape.n_layers} of a token, lm_head "
              f"excluded) through the fp64 C oracle; {args.steps} steps in {dt:.1f} s")
    return {"metric": METRIC, "value": round(tok_s, 4), "unit": "tok/s", "impl": "reference",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per_layer * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": f"llama3-8b-shaped Q8_0, B={B} sessions at ctx {PREFILL}..{PREFILL + WINDOW - 1}",
                       "batch": B},
            "cpu_baseline": {"value": round(tok_s, 4), "unit": "tok/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(tok_s, 4), "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=512)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--batch", type=int, default=8)
    ap.add_argument("--impl", default="kd", choices=["kd", "reference"])
    ap.add_argument("--no-sweep", dest="sweep", action="store_false")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", dest="workloads", action="store_false",
                    help="skip the long-context, isolated-mmvq and isolated-attention measurements")
    ap.add_argument("--op", choices=["mmvq", "attn", "long", "step", "timeline"],
                    help="time one kernel family in isolation, the long-context step, the 8B-shaped step "
                         "at --layers depth, or the per-kernel in-step timeline of the 8B-shaped step")
    ap.add_argument("--layers", type=int, default=2, help="decoder layers of --op step")
    ap.add_argument("--rows", type=int, default=4096)
    ap.add_argument("--cols", type=int, default=14336)
    ap.add_argument("--m", type=int, default=8)
    ap.add_argument("--cap", type=int, default=32768)
    ap.add_argument("--kv-q8", action="store_true", help="--op attn / long / timeline: the Q8_0 KV cache")
    ap.add_argument("--long", action="store_true", help="--op timeline: the long-context case")
    args = ap.parse_args()
    if args.op:
        r = {"mmvq": run_op_mmvq, "attn": run_op_attn, "long": run_op_long, "step": run_op_step,
             "timeline": run_op_timeline}[args.op](args)
        print(json.dumps(r), flush=True)
        return
    args.warmup = max(args.warmup, 3)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        torch.distributed.init_process_group("nccl")
    r = run_kd(args, rank, world)
    if rank == 0:
        shape = synth.LLAMA3_8B
        out = {
            "metric": METRIC, "value": round(r["value"], 2), "unit": "tok/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(r["ms"] / args.steps, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16xq8_0->f32", "data": "synthetic",
            "config": {"workload": f"llama3-8b-shaped Q8_0 decode, B={args.batch} sessions, KV fp16 pre-filled to "
                                   f"{PREFILL}, positions {PREFILL}..{PREFILL + WINDOW - 1} cycling",
                       "batch": args.batch, "prefill": PREFILL, "capacity": CAPACITY,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": "inputs larger than L2: 7.97 GB of Q8_0 weights streamed per step"},
            "hbm_gbs": round(r["gbs"], 1),
            "hbm_frac_of_peak": round(r["gbs"] / r["peak"], 4),
            "peak_hbm_gbs": r["peak"], "peak_source": r["peak_kind"],
            "e2e": r["e2e"], "roofline": r["roofline"], "batch_sweep": r["sweep"],
            "cpu_baseline": r["cpu"], "clocks": r["clocks"],
            "gpu_launches": int(round(r["launches_per_step"] * args.steps)),
            "kernel_time_share": r["shares"], "device_status": r["status"],
            "workloads": r["workloads"],
        }
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
