"""Benchmark of the quantised-KV decode step on GB300.

One step = for each of R independent layer caches (R chosen so their bytes
exceed L2 several times): append one token's K/V (q8_0 / q5_1 quantise +
commit), decode attention of one query row over the whole cache (split +
merge kernels), and truncate the appended row again (rollback to
snapshot_len + 0), so every step sees the same length.  Inputs are resident in
HBM before the timed region.  The decode time is what the decode adds to the
step: the captured K-step graph minus the same graph without the decodes, both
timed by CUDA events around the replay on the launching stream.

`value` is GB/s of quantised KV read by the decode (algorithmic bytes: every
visible row x (K 34 + V 24 bytes per 32 elements, or 32 + 32 with
--kv-format e4m3)), summed over all ranks.
`e2e` repeats the step through the same public API with the step's inputs
copied from pinned host memory and the attention output copied back inside
the timed region.  `--impl reference` times the fp64 CPU oracle on a bounded
sample of the same workload.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
       [--also NAME,...|none] [--layers R] [--kv-format q8_0/q5_1|e4m3] [--t T]
       [--softcap C] [--rollback host|device] [--impl kvq|reference]

The headline line is --workload (ctx32k by default); the workloads named by
--also (batch64 by default) are measured in the same run and reported under
"workloads", each with its own value, roofline, e2e and CPU baseline.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from quantized_kv_cache_08_gb300 import build as kbuild  # noqa: E402
from quantized_kv_cache_08_gb300.inputs import workload  # noqa: E402

METRIC = "decode-attn GB/s of quantized KV read (fraction of HBM peak); tokens/s"
L2_BYTES = 129 * 1024 * 1024


FORMATS = {"q8_0/q5_1": ("K q8_0 / V q5_1", 34 + 24), "e4m3": ("K, V fp8 e4m3", 32 + 32)}


def kv_bytes_per_row(wl, fmt="q8_0/q5_1"):
    kb = wl.n_kv * wl.head_dim // 32
    return kb * FORMATS[fmt][1]


def decode_lengths(wl):
    """Lengths at decode.  A ring holds the same visible rows at any length
    past window + T, so its caches fill to twice the window instead of the
    workload's final length (the decode then reads the same bytes)."""
    lens = wl.lengths()
    if wl.ring:
        lens = [min(L, 2 * wl.window) for L in lens]
    return lens


def visible_rows(wl, L):
    """Rows a T-row decode reads: the union of the query rows' windows."""
    if wl.window:
        return L - max(0, L - wl.T + 1 - wl.window)
    return L


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_source_hash():
    """Hash of the CUDA sources with comments removed and whitespace collapsed,
    so that recorded counters stay valid across comment-only edits and no
    longer."""
    h = hashlib.sha256()
    for f in sorted(os.listdir(os.path.join(ROOT, "quantized_kv_cache_08_gb300", "csrc"))):
        with open(os.path.join(ROOT, "quantized_kv_cache_08_gb300", "csrc", f)) as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        src = " ".join(src.split())
        h.update(f.encode() + b"\0" + src.encode())
    return h.hexdigest()[:16]


def traffic_key(name, fmt, args):
    """Key of a run's recorded ncu traffic: the workload, plus every option
    that changes the kernel or the shape (format, soft-capping, query rows)."""
    key = name if fmt == "q8_0/q5_1" else f"{name}:{fmt}"
    if args.softcap > 0:
        key += ":softcap"
    if args.t:
        key += f":T{args.t}"
    return key


def recorded_traffic(name):
    """dram bytes per decode launch from a committed ncu summary, if it was
    taken on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(name)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_decode")


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"kvq_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 7:
                    continue
                try:
                    sm.append(float(parts[0]))
                    mx.append(float(parts[1]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[3:7]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def max_over_ranks(x, world):
    """Largest value of x over ranks (the job's time); x on every rank."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def bench_workload(args):
    """The named workload, with its query rows per step overridden by --t."""
    return workload(args.workload, **({"T": args.t} if args.t else {}))


DTYPE = ("k.q: int16 queries x int8 codes (dp2a, int32 sums, f32 per block); "
         "p.v: f32 (packed FMA)")


def measure(args, name, world, rank, local):
    """One workload: build R layer caches, time the captured step, return the
    workload's result (value, roofline, e2e, clocks, config)."""
    from quantized_kv_cache_08_gb300.cache import KVCache

    dev = torch.device("cuda", local)
    wl = workload(name, **({"T": args.t} if args.t else {}))
    T = wl.T
    lens = decode_lengths(wl)
    fmt = args.kv_format
    row_bytes = kv_bytes_per_row(wl, fmt)
    vis = [visible_rows(wl, L) for L in lens]
    footprint = sum(vis) * row_bytes
    R = args.layers or min(8, max(1, math.ceil(3 * L2_BYTES / footprint)))
    flush = R * footprint < 3 * L2_BYTES
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.set_stream(stream)
    sinks = wl.sink_logits()
    sinks_d = None if sinks is None else sinks.to(dev)
    scratch = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) if flush else None
    device_rollback = args.rollback == "device"
    # rows past the step's length: the e2e legs run their steps before the
    # host mirror is read back (device rollback), each step appending T rows
    spare = T * (4 * (args.steps + args.warmup) + 8) if device_rollback else T

    # --- build R layer caches holding len-T rows each (prefill, untimed);
    # a ring fills with T-row steps, a flat cache with 64-row chunks
    caches = []
    for r in range(R):
        if wl.ring:
            c = KVCache(wl.n_seq, wl.n_kv, wl.head_dim, wl.n_q, max_t=T, window=wl.window, ring=True,
                        fmt=fmt)
        else:
            c = KVCache(wl.n_seq, wl.n_kv, wl.head_dim, wl.n_q, max_t=max(64, T), max_rows=max(lens) + spare,
                        window=wl.window, fmt=fmt)
        if args.softcap > 0:
            c.set_softcap(args.softcap)
        chunk = T if wl.ring else 64
        for b, L in enumerate(lens):
            k, v = wl.kv(b + 1000 * r + 100000 * rank, 0, L - T + 64 * T)
            kd, vd = k.to(dev), v.to(dev)
            for t0 in range(0, L - T, chunk):
                t1 = min(L - T, t0 + chunk)
                c.append(kd[t0:t1].unsqueeze(0), vd[t0:t1].unsqueeze(0), seq_ids=[b])
            if wl.ring and r == 0:
                # the step appends T rows and truncates them again: fill on
                # until that append needs no rebase and the window of the
                # truncated length is still resident, then every layer
                # fills to that length
                n = L - T
                while c.ring_headroom(T) < 1 or n - T + 1 - wl.window < c.bases()[b]:
                    c.append(kd[n:n + T].unsqueeze(0), vd[n:n + T].unsqueeze(0), seq_ids=[b])
                    n += T
                lens[b] = n + T
        caches.append(c)
    base_len = [L - T for L in lens]
    # --- per-layer step inputs, resident on the device
    k_new, v_new, qs = [], [], []
    for r in range(R):
        kk = torch.stack([wl.kv(b + 1000 * r + 100000 * rank, L - T, L)[0] for b, L in enumerate(lens)])
        vv = torch.stack([wl.kv(b + 1000 * r + 100000 * rank, L - T, L)[1] for b, L in enumerate(lens)])
        k_new.append(kk.to(dev))
        v_new.append(vv.to(dev))
        qs.append(wl.q(r + 7 * rank, T=T).to(dev))
    # the layers' outputs side by side in one buffer: the step's result
    out_all = torch.empty(R, wl.n_seq, T, wl.n_q, wl.head_dim, dtype=torch.float32, device=dev)
    outs = list(out_all.unbind(0))
    accept0 = torch.zeros(wl.n_seq, dtype=torch.int32, device=dev)

    def rollback(c):
        """Back to the snapshot: T draft rows, none accepted."""
        if device_rollback:
            c.truncate_device(accept0, T)
        else:
            c.truncate(base_len)

    torch.cuda.synchronize()

    def step(events=None, decode=True):
        if scratch is not None:
            scratch.zero_()                 # inputs smaller than L2: flush it every step
        for r, c in enumerate(caches):
            c.append(k_new[r], v_new[r])
            if events is not None:
                events[r][0].record(stream)
            if decode:
                c.decode(qs[r], sinks=sinks_d, out=outs[r])
            if events is not None:
                events[r][1].record(stream)
            rollback(c)

    def sync_all():
        torch.cuda.synchronize()
        if device_rollback:
            for c in caches:
                c.sync_len()

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        return g

    def replay_ms(g):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    # eager warm-up (kernel attributes, lazy module loads), then capture.  The
    # counters live on the device, so the captured append / decode / rollback
    # replay with the right lengths.  The decode time is what the decode adds
    # to the step: the K-step graph (the timed region) minus the same graph
    # without the decodes, both timed by CUDA events around the replay on the
    # launching stream.  Event nodes inside a graph cost microseconds each,
    # so the per-decode event brackets and a graph of back-to-back decodes are
    # reported beside it as cross-checks only.
    step()
    sync_all()
    g_warm = capture(step)
    g_timed = capture(lambda: [step() for _ in range(args.steps)])
    g_nodec = capture(lambda: [step(decode=False) for _ in range(args.steps)])
    try:   # event record nodes inside the graph (torch >= 2.6 'external' events)
        ev = [[[torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
               for _ in range(R)] for _ in range(args.steps)]
        g_ev = capture(lambda: [step(ev[k]) for k in range(args.steps)])
    except TypeError:
        ev, g_ev = None, None

    def dec_only():
        for _ in range(args.steps):
            for r, c in enumerate(caches):
                c.decode(qs[r], sinks=sinks_d, out=outs[r])
    g_dec = capture(dec_only)
    sync_all()
    for _ in range(args.warmup):
        g_warm.replay()
    torch.cuda.synchronize()
    barrier(world)
    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.3)
    step_ms = statistics.median(replay_ms(g_timed) for _ in range(3))
    clk = clocks.stop()
    barrier(world)
    nodec_ms = statistics.median(replay_ms(g_nodec) for _ in range(3))
    g_dec.replay()
    dec_only_ms = max_over_ranks(replay_ms(g_dec), world)
    bracket_ms = None
    if g_ev is not None:
        g_ev.replay()
        torch.cuda.synchronize()
        bracket_ms = max_over_ranks(sum(a.elapsed_time(b) for evk in ev for a, b in evk), world)
    total_ms = max_over_ranks(step_ms, world)
    dec_ms = max_over_ranks(step_ms - nodec_ms, world)
    timing = ("decode = CUDA-graph replay of K steps minus the same K steps without the decode, "
              "CUDA events around each replay on the launching stream")
    sync_all()
    for c in caches:
        if c.device_error() != 0:
            raise SystemExit("device error word set during the benchmark")

    kv_bytes_step = R * footprint                       # per rank
    decodes = args.steps * R
    value = world * kv_bytes_step * args.steps / (dec_ms * 1e-3) / 1e9
    tokens_per_s = world * wl.n_seq * T * decodes / (dec_ms * 1e-3)   # query rows per second
    achieved = kv_bytes_step * args.steps / (dec_ms * 1e-3) / 1e9  # per GPU
    peak, peak_src = measured_peak()

    # --- end to end through the public API: the step's inputs (K, V rows and
    # queries, in their own dtypes) in one pinned host buffer copied in with
    # one copy, the step's outputs (every layer's) copied out with one copy
    segs, off = [], 0
    for x in k_new + v_new + qs:
        nb = x.numel() * x.element_size()
        segs.append((off, nb, x))
        off += (nb + 255) // 256 * 256
    host_in = torch.empty(off, dtype=torch.uint8).pin_memory()
    dev_in = torch.empty(off, dtype=torch.uint8, device=dev)
    ins = []
    for o, nb, x in segs:
        host_in[o:o + nb].copy_(x.reshape(-1).view(torch.uint8).cpu())
        ins.append(dev_in[o:o + nb].view(x.dtype).view(x.shape))
    dk, dv, dq = ins[:R], ins[R:2 * R], ins[2 * R:]
    pin_o = torch.empty(out_all.shape, dtype=out_all.dtype).pin_memory()

    def e2e_step():
        dev_in.copy_(host_in, non_blocking=True)
        for r, c in enumerate(caches):
            c.append(dk[r], dv[r])
            c.decode(dq[r], sinks=sinks_d, out=outs[r])
            rollback(c)
        pin_o.copy_(out_all, non_blocking=True)

    # eager: every call from Python, as a caller without graphs makes them
    for _ in range(args.warmup):
        e2e_step()
    sync_all()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_eager_ms = max_over_ranks(e0.elapsed_time(e1), world)
    sync_all()
    # captured: the same public calls and copies (pinned host -> device inputs,
    # device -> pinned host outputs) replayed as one CUDA graph of K steps
    g_e2e = capture(lambda: [e2e_step() for _ in range(args.steps)])
    for _ in range(args.warmup):
        g_e2e.replay()
    sync_all()
    barrier(world)
    e2e_ms = max_over_ranks(statistics.median(replay_ms(g_e2e) for _ in range(3)), world)
    sync_all()
    h2d = sum(nb for _, nb, _ in segs)
    d2h = pin_o.numel() * pin_o.element_size()
    e2e_value = world * kv_bytes_step * args.steps / (e2e_ms * 1e-3) / 1e9

    extra = ""
    if wl.window:
        extra += f", window {wl.window}" + (f" over a ring of {caches[0].rows} rows" if wl.ring else "")
    if sinks is not None:
        extra += ", a sink logit per Q head"
    if args.softcap > 0:
        extra += f", scores soft-capped at {args.softcap:g}"
    cfg = {"workload": f"{wl.name}: {wl.n_seq} seq, {wl.n_q} Q / {wl.n_kv} KV heads, head_dim "
                       f"{wl.head_dim}, {sum(lens)} rows at decode, T={T}{extra}, q {wl.q_dtype}, "
                       f"{FORMATS[fmt][0]}",
           "layers": R, "rows_total": sum(lens), "rows_visible": sum(vis),
           "kv_bytes_per_decode": footprint,
           "step": (f"per layer: append {T} row(s) + decode + rollback to the snapshot "
                    f"({'device-side accepted counts' if device_rollback else 'host lengths'})"),
           "l2": (f"L2 flushed every step ({2 * L2_BYTES // 2**20} MiB write), {R} layer caches"
                  if flush else
                  f"inputs larger than L2: {R} layer caches, {R * footprint / 1e6:.0f} MB rotated")}
    res = {
        "value": round(value, 2), "unit": "GB/s",
        "ms_per_step": round(total_ms / args.steps, 4),
        "config": cfg,
        "tokens_per_s": round(tokens_per_s, 1),
        "decode_ms_per_layer": round(dec_ms / decodes, 5),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": recorded_traffic(traffic_key(wl.name, fmt, args)),
                     "peak_source": peak_src,
                     "kernel": "kvq decode (split + merge)"},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms / args.steps, 4),
                "how": "K steps of the public calls with their pinned-host copies (the step's K, V "
                       "and queries in one buffer in, every layer's output in one buffer back), captured as one CUDA graph and "
                       "replayed; the whole step's time (copies, append, decode, rollback) divides the "
                       "decode's bytes",
                "eager_value": round(world * kv_bytes_step * args.steps / (e2e_eager_ms * 1e-3) / 1e9, 2)},
        # append, split, merge, rollback per layer and step
        "gpu_launches": 4 * R * args.steps,
        "timing": timing,
        "decode_only_ms_per_layer": round(dec_only_ms / decodes, 5),
        "decode_event_bracket_ms_per_layer": None if bracket_ms is None else round(bracket_ms / decodes, 5),
        "step_without_decode_ms_per_layer": round(nodec_ms / decodes, 5),
        "clocks": clk,
    }
    if wl.ring:
        res["ring_growth"] = ring_growth(caches[0], wl, k_new[0], v_new[0], qs[0], sinks_d, outs[0],
                                         args, row_bytes, vis[0], world)
    if rank == 0 and world == 1:
        res["cpu_baseline"] = cpu_baseline(wl, lens, sinks=sinks, fmt=fmt, softcap=args.softcap)
    del caches, g_warm, g_timed, g_nodec, g_ev, g_dec, g_e2e
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def ring_growth(c, wl, k1, v1, q1, sinks_d, out, args, row_bytes, vis, world, steps=256):
    """A ring that keeps growing: eager append + decode steps with no rollback,
    so every 32nd append rebases the ring (moves the live window to row 0)
    inside the timed region; CUDA events around the K steps."""
    T = wl.T
    for _ in range(8):
        c.append(k1, v1)
        c.decode(q1, sinks=sinks_d, out=out)
    torch.cuda.synchronize()
    b0 = c.bases()[0]
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        c.append(k1, v1)
        c.decode(q1, sinks=sinks_d, out=out)
    e1.record()
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), world)
    rebases = (c.bases()[0] - b0) // 32
    return {"steps": steps, "ms_per_step": round(ms / steps, 5),
            "rebases": int(rebases),
            "value": round(world * vis * row_bytes * steps / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "how": f"eager append of {T} row(s) + decode per step, the length growing (no rollback), a ring "
                   "rebase every 32 appends inside the timed region; the decode's bytes over the whole step"}


def run_kvq(args, world, rank, local):
    kbuild.build()
    torch.cuda.set_device(local)
    res = measure(args, args.workload, world, rank, local)
    line = {"metric": METRIC, "value": res.pop("value"), "unit": res.pop("unit"), "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": res.pop("ms_per_step"),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": DTYPE,
            "data": "synthetic"}
    line.update(res)
    extras = [w for w in (args.also.split(",") if args.also and args.also != "none" else [])
              if w and w != args.workload]
    if extras:
        line["workloads"] = {w: measure(args, w, world, rank, local) for w in extras}
        line["gpu_launches"] += sum(v["gpu_launches"] for v in line["workloads"].values())
    return line


def cpu_baseline(wl, lens, budget_s=12.0, sinks=None, fmt="q8_0/q5_1", softcap=0.0):
    """The fp64 oracle, as it stands, on a bounded sample of the workload: the
    decode of one layer for the first sequence (quantise its rows once, then
    dequantise + attend per repetition)."""
    from oracle import kvq_oracle as O

    L = lens[0]
    k, v = wl.kv(0, 0, L)
    ora = O.OracleKvCache(1, wl.n_kv, wl.head_dim, window=wl.window, fmt=fmt)
    ora.append(k.unsqueeze(0).numpy(), v.unsqueeze(0).numpy())
    q = wl.q(0)[:1].float().numpy().astype("float64")
    sk = None if sinks is None else sinks.double().numpy()
    reps, t_total = 0, 0.0
    while t_total < budget_s and reps < 20:
        t = time.perf_counter()
        ora.decode(q, sinks=sk, softcap=softcap)
        t_total += time.perf_counter() - t
        reps += 1
    gbs = reps * visible_rows(wl, L) * kv_bytes_per_row(wl, fmt) / t_total / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{reps} fp64 decodes of 1 sequence x {visible_rows(wl, L)} visible rows ({wl.name}), "
                      f"numpy with its default BLAS threading, {t_total:.1f} s"}


def run_reference(args, world, rank):
    """The oracle as the reference arm: K timed steps, each a bounded sample."""
    if rank != 0:
        return None
    wl = bench_workload(args)
    lens = decode_lengths(wl)
    base = cpu_baseline(wl, lens, budget_s=max(2.0, 60.0 / max(1, args.steps + args.warmup)),
                        sinks=wl.sink_logits(), fmt=args.kv_format, softcap=args.softcap)
    return {"impl": "reference", "metric": METRIC, "value": base["value"], "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": wl.name, "T": wl.T, "kv_format": args.kv_format,
                                            "softcap": args.softcap, "sample": base["sample"]},
            "cpu_baseline": base,
            "e2e": {"value": base["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------ ncu summaries

_UNITS = {"byte": 1, "kbyte": 1e3, "mbyte": 1e6, "gbyte": 1e9, "ns": 1e-3, "nsecond": 1e-3, "us": 1.0,
          "usecond": 1.0, "ms": 1e3, "msecond": 1e3, "s": 1e6, "second": 1e6}


def _short_kernel(name):
    """Kernel name without return type, namespaces and parameter list."""
    name = re.sub(r"^void ", "", name).replace("<unnamed>", "anon").replace("unnamed>", "anon").replace("(anonymous namespace)", "anon")
    depth, cut = 0, len(name)
    for i, ch in enumerate(name):
        if ch == "<":
            depth += 1
        elif ch == ">":
            depth -= 1
        elif ch == "(" and depth == 0:
            cut = i
            break
    name = name[:cut]
    return re.sub(r"^(?:[A-Za-z_]\w*::)+", "", name)


def read_ncu_csv(path):
    """Launches of an `ncu --csv --log-file` log: [(id, kernel, {metric: value})],
    bytes in bytes and times in microseconds."""
    import csv
    with open(path) as fh:
        lines = [ln for ln in fh if not ln.startswith("==")]
    rows = list(csv.reader(lines))
    hdr = next(i for i, r in enumerate(rows) if "Metric Name" in r)
    cols = {name: j for j, name in enumerate(rows[hdr])}
    launches = {}
    for r in rows[hdr + 1:]:
        if len(r) < len(cols):
            continue
        lid = int(r[cols["ID"]])
        unit = r[cols["Metric Unit"]].strip().lower()
        try:
            v = float(r[cols["Metric Value"]].replace(",", "")) * _UNITS.get(unit, 1.0)
        except ValueError:
            continue
        e = launches.setdefault(lid, (r[cols["Kernel Name"]], {}))
        e[1][r[cols["Metric Name"]]] = v
    return [(lid, k, m) for lid, (k, m) in sorted(launches.items())]


def _decode_role(kernel):
    if "merge" in kernel:
        return "merge_kernel"
    if "stream_kernel" in kernel or "split_kernel" in kernel:
        return "split_kernel"
    return None


def record_ncu_traffic(args, path, how):
    """Average DRAM bytes per launch of the decode's split and merge kernels in
    an ncu log, written to profiles/traffic.json under this run's key, with
    the kernel-source hash they belong to."""
    wl = bench_workload(args)
    fmt = args.kv_format
    sums = {}
    for _, kernel, m in read_ncu_csv(path):
        role = _decode_role(kernel)
        if role is None or "dram__bytes_read.sum" not in m:
            continue
        acc = sums.setdefault(role, [0, 0.0, 0.0, kernel])
        acc[0] += 1
        acc[1] += m["dram__bytes_read.sum"]
        acc[2] += m.get("dram__bytes_write.sum", 0.0)
    if "split_kernel" not in sums:
        raise SystemExit(f"{path}: no split-kernel launch with dram__bytes_read.sum")
    alg = sum(visible_rows(wl, L) for L in decode_lengths(wl)) * kv_bytes_per_row(wl, fmt)
    key = traffic_key(wl.name, fmt, args)
    rec = {"source_hash": kernel_source_hash(), "algorithmic_bytes_per_decode": alg, "how": how}
    total = 0
    for role, (n, rd, wr, kernel) in sums.items():
        rec[role] = {"kernel": _short_kernel(kernel), "launches": n, "dram_bytes_read": int(round(rd / n)),
                     "dram_bytes_write": int(round(wr / n))}
        total += rec[role]["dram_bytes_read"] + rec[role]["dram_bytes_write"]
    rec["dram_bytes_per_decode"] = total
    out = os.path.join(ROOT, "profiles", "traffic.json")
    d = {}
    if os.path.exists(out):
        with open(out) as fh:
            d = json.load(fh)
    d[key] = rec
    with open(out, "w") as fh:
        json.dump(d, fh, indent=1, sort_keys=True)
        fh.write("\n")
    return key, rec


def launch_table(path):
    """Markdown launch list of an ncu log of gpu__time_duration.sum: launches,
    total and mean time and share per kernel."""
    per = {}
    for _, kernel, m in read_ncu_csv(path):
        t = m.get("gpu__time_duration.sum")
        if t is None:
            continue
        e = per.setdefault(_short_kernel(kernel), [0, 0.0])
        e[0] += 1
        e[1] += t
    tot = sum(v[1] for v in per.values())
    out = ["| kernel | launches | total µs | share | mean µs |", "|---|---|---|---|---|"]
    for k, (n, t) in sorted(per.items(), key=lambda kv: -kv[1][1]):
        out.append(f"| `{k}` | {n} | {t:.1f} | {100 * t / tot:.1f}% | {t / n:.2f} |")
    out.append(f"| total | {sum(v[0] for v in per.values())} | {tot:.1f} | 100% | |")
    return "\n".join(out)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="ctx32k")
    ap.add_argument("--layers", type=int, default=0)
    ap.add_argument("--kv-format", default="q8_0/q5_1", choices=sorted(FORMATS),
                    help="K/V storage: q8_0 K with q5_1 V (default), or FP8 E4M3 K and V")
    ap.add_argument("--t", type=int, default=0,
                    help="query rows per step (appended, decoded causally, truncated); 0 = the workload's")
    ap.add_argument("--softcap", type=float, default=0.0,
                    help="score soft-capping c (s -> c tanh(s / c)); 0 = off")
    ap.add_argument("--also", default="batch64",
                    help="comma-separated workloads measured in the same run, reported under "
                         "'workloads' (none: only --workload)")
    ap.add_argument("--rollback", default="host", choices=["host", "device"],
                    help="how each step rolls back to the snapshot: host lengths (kvq_truncate) or "
                         "accepted counts on the device (kvq_truncate_device)")
    ap.add_argument("--impl", default="kvq", choices=["kvq", "reference"])
    ap.add_argument("--ncu-traffic", metavar="CSV",
                    help="record the decode kernels' DRAM bytes per launch from an ncu --csv log "
                         "(dram__bytes_read.sum, dram__bytes_write.sum) in profiles/traffic.json under "
                         "this run's workload and options, then exit; --ncu-how gives the command")
    ap.add_argument("--ncu-how", default="", help="the ncu command that wrote the --ncu-traffic log")
    ap.add_argument("--ncu-launches", metavar="CSV",
                    help="print the launch list (launches, time, share per kernel) of an ncu --csv log "
                         "of gpu__time_duration.sum as a markdown table, then exit")
    args = ap.parse_args()
    if args.ncu_traffic:
        key, rec = record_ncu_traffic(args, args.ncu_traffic, args.ncu_how)
        print(json.dumps({key: rec}, indent=1))
        return
    if args.ncu_launches:
        print(launch_table(args.ncu_launches))
        return
    if args.warmup < 3:
        args.warmup = 3
    if not 0 <= args.t <= 512:
        ap.error("--t must be in [1, 512] (0 = the workload's own)")
    if args.softcap < 0:
        ap.error("--softcap must be >= 0")
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        line = run_reference(args, world, rank)
    else:
        line = run_kvq(args, world, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
