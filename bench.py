"""Benchmark of the batched GDN verify + commit transaction on GB300.

One step = one MTP verify cycle of the whole stack: gdn_conv_verify for each of
the 30 GDN layers, then one grouped gdn_commit for all layers with keep[]
re-drawn every cycle (B=8 rows, T=2 positions, H_k=16, H_v=32, d=128, rows 6-7
inactive).  The commit strategy defaults to DEFERRED: the commit records keep
and shifts the conv windows, and each layer's next verify applies the state
update while it holds the state anyway (--mode recompute|snapshot for the
eager strategies).  The metric is row-tokens/s (B*T verified positions per cycle
divided by the cycle time) together with the achieved HBM bandwidth against
the measured GB300 copy peak.

Inputs are synthetic (seeded ``synth`` draws, x/g/beta from a pool of 16
cycles, keep[] fresh every cycle) and resident in HBM before timing starts;
the 480 MiB state stack is larger than the 129 MB L2, so no flush is needed.
Each cycle is one captured CUDA graph of the C-ABI calls.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
        [--mode recompute|snapshot|deferred] [--B 8 --T 2 --layers 30] [--no-cpu-baseline]
Under torchrun (N > 1) every rank runs its own cohort (weak scaling, no
collective on the data path) and rank 0 prints the max-over-ranks result.
"""
from __future__ import annotations

import argparse
import concurrent.futures
import hashlib
import json
import os
import shutil
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GDN verify+commit row-tokens/s and achieved HBM GB/s vs GB300 peak (1 GPU)"
UNIT = "row-tokens/s"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = {
    "commit": ["speculative_decode_gated_gdn_gb300/csrc/commit.cu",
               "speculative_decode_gated_gdn_gb300/csrc/gdn_common.cuh"],
    "verify": ["speculative_decode_gated_gdn_gb300/csrc/verify.cuh",
               "speculative_decode_gated_gdn_gb300/csrc/gdn_common.cuh"],
}


MODES = {"recompute": 0, "snapshot": 1, "deferred": 2}  # GDN_COMMIT_* of the C ABI


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1024)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--mode", default="deferred", choices=list(MODES))
    ap.add_argument("--B", type=int, default=8)
    ap.add_argument("--T", type=int, default=2)
    ap.add_argument("--layers", type=int, default=30)
    ap.add_argument("--inactive", type=str, default=None,
                    help="comma list of inactive rows (default: rows 6-7 at B=8, else the last B/4)")
    ap.add_argument("--seed", type=int, default=2)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--workload", default="cycle", choices=["cycle", "prefill", "accept"],
                    help="cycle: the verify+commit headline; prefill: chunked state priming of one row; "
                         "accept: the on-device greedy acceptance kernel alone")
    ap.add_argument("--accept", action="store_true",
                    help="cycle: take keep from gdn_accept_greedy on synthetic logits (verify + accept + commit "
                         "per graph) instead of drawing it")
    ap.add_argument("--V", type=int, default=151936, help="vocabulary size for acceptance")
    ap.add_argument("--gated", action="store_true",
                    help="cycle: verify through gdn_conv_verify_gated (gated RMSNorm of the output fused in)")
    ap.add_argument("--L", type=int, default=4096, help="prompt length for --workload prefill")
    return ap.parse_args()


# ---------------------------------------------------------------- geometry
def workload(args):
    from speculative_decode_gated_gdn_gb300 import synth
    geom = synth.Geometry(B=args.B, T=args.T, H_k=16, H_v=32, d=128)
    if args.inactive is not None:
        inactive = tuple(int(v) for v in args.inactive.split(",") if v != "")
    elif args.B == 8:
        inactive = (6, 7)
    else:
        inactive = tuple(range(args.B - args.B // 4, args.B))
    return geom, inactive


def config_dict(args, geom, inactive):
    acc = getattr(args, "accept", False)
    keep_txt = (f"keep from on-device greedy acceptance over V={args.V} (drafts planted so keep~U{{1..{geom.T}}}), "
                f"verify+accept+commit per graph" if acc else f"keep~U{{0..{geom.T}}} per cycle")
    return {
        "workload": (f"GDN verify+commit cycle: B={geom.B} T={geom.T} H_k={geom.H_k} H_v={geom.H_v} "
                     f"d={geom.d} x {args.layers} layers, {keep_txt}, "
                     f"inactive rows {list(inactive)}"),
        "keep_source": "gdn_accept_greedy" if acc else "drawn",
        "output": "gated RMSNorm fused (gdn_conv_verify_gated)" if getattr(args, "gated", False) else "o",
        "B": geom.B, "T": geom.T, "H_k": geom.H_k, "H_v": geom.H_v, "d": geom.d,
        "layers": args.layers, "commit_mode": args.mode, "inactive_rows": list(inactive),
        "l2": f"no flush: state stack {args.layers * geom.B * geom.H_v * geom.d * geom.d * 4 / 2**20:.0f} MiB "
              f"> 129 MB L2",
        "parallelism": "replicas" if args.gpus > 1 else "single GPU",
    }


def state_row_bytes(geom):
    return geom.H_v * geom.d * geom.d * 4


def verify_bytes(geom, n_active, mode="recompute", n_apply=0):
    """Algorithmic bytes of one verify launch: state read once per active row,
    raw inputs, taps, conv window read + new ring slots, gates, outputs; in
    SNAPSHOT mode the T snapshots written per active row; in DEFERRED mode the
    committed state written back for the n_apply rows whose commit it applies."""
    C = geom.C
    b = (state_row_bytes(geom) * n_active + n_active * geom.T * C * 2 + C * 4 * 2
         + n_active * (3 + geom.T) * C * 2 + n_active * geom.T * geom.H_v * 4 * 2
         + geom.B * geom.T * geom.H_v * geom.d * 2)
    if mode == "snapshot":
        b += geom.T * state_row_bytes(geom) * n_active
    if mode == "deferred":
        b += state_row_bytes(geom) * n_apply
    return b


def ring_shift_bytes(geom, n_keep, n_layers):
    """Conv-window shift of the commit: three slots read and written per kept row."""
    return 2 * 3 * geom.C * 2 * n_keep * n_layers


def commit_bytes(geom, n_keep, n_layers, mode="recompute"):
    """Algorithmic bytes of one grouped commit launch.  RECOMPUTE: read S_0 and
    write S_keep for every (layer, row) with keep' >= 1; SNAPSHOT: read the
    snapshot S_keep and write it; DEFERRED: only the keep record and the window
    shift (the state update moves into the next verify)."""
    state = 0 if mode == "deferred" else 2 * state_row_bytes(geom) * n_keep * n_layers
    return state + ring_shift_bytes(geom, n_keep, n_layers)


def path_min_bytes(geom, n_active, n_keep, n_layers):
    """The least HBM traffic of a cycle whatever the commit strategy: every
    active row's state read once, every kept row's state written once, plus
    the inputs, outputs and conv windows."""
    per_layer = verify_bytes(geom, n_active) + state_row_bytes(geom) * n_keep
    return n_layers * per_layer + ring_shift_bytes(geom, n_keep, n_layers)


# ---------------------------------------------------------------- environment
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_seed(seed, rank):
    """Each rank verifies its own cohort: disjoint seeded draws per rank."""
    return seed + 1000 * rank


def max_over_ranks(ms, device, world):
    """The job's elapsed time is its slowest rank's: max of the per-rank times."""
    if world == 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, units_per_rank_step, step_ms):
    """Whole-job throughput: every rank processes its own units each step."""
    return world * units_per_rank_step / (step_ms * 1e-3)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id: str | None):
        self.device_id = device_id
        self.proc = None
        self.lines: list[str] = []
        self.t0 = self.t1 = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def __enter__(self):
        exe = shutil.which("nvidia-smi")
        if exe:
            cmd = [exe, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "20"]
            if self.device_id:
                cmd += ["-i", self.device_id]
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
            time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.reader.join(timeout=2)

    def summary(self):
        if not self.proc:
            return None
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        import datetime
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                if self.t0 is not None and not (self.t0 - 0.02 <= ts <= self.t1 + 0.02):
                    continue
                sm.append(float(parts[2]))
                smax.append(float(parts[3]))
                power.append(float(parts[4]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[6:10]):
                if flag.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power), "window": "timed region only"}


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_hash(kind):
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kind, workload_key):
    """dram bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (null otherwise)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[kind][workload_key]
    except Exception:
        return None
    if rec.get("source_hash") != source_hash(kind):
        return None
    return rec.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- CPU oracle
def oracle_layer_cycle(orc, geom, st, cy, layer, active, keep):
    """One layer's verify + commit on the CPU oracle (fp64)."""
    from speculative_decode_gated_gdn_gb300 import synth
    ring = st["ring"][layer]
    offsets = st["offsets"]
    win = np.empty((geom.B, geom.C, 3))
    for b in range(geom.B):
        for i in range(3):
            win[b, :, i] = synth.bf16_to_f32(ring[b, i])  # committed window: slots 0..2
    x = synth.bf16_to_f32(cy["x"][layer]).astype(np.float64)
    w = synth.bf16_to_f32(st["conv_w"][layer]).astype(np.float64)
    S = st["state"][layer].copy()
    o, Sall = orc.verify(x, w, win, cy["g"][layer], cy["beta"][layer], S, active, H_k=geom.H_k, act=geom.act)
    off = offsets.copy()
    orc.commit(keep, active, Sall, x, S, win, off)
    return o


def run_oracle_sample(geom, inactive, n_layers, seconds, max_layer_cycles=None, seed=2):
    """Time the oracle on a bounded sample of layer-cycles using all host cores
    (threads over independent layers; the C oracle runs without the GIL)."""
    import oracle
    from speculative_decode_gated_gdn_gb300 import synth
    orc = oracle.default()
    sample_layers = min(n_layers, 4)
    st = synth.layer_state(geom, seed, sample_layers)
    cy = synth.cycle_inputs(geom, seed, 0, sample_layers)
    active = synth.active_mask(geom.B, inactive)
    keep = cy["keep"]
    cores = os.cpu_count() or 1
    done = 0
    t0 = time.perf_counter()
    with concurrent.futures.ThreadPoolExecutor(max_workers=cores) as ex:
        while True:
            futs = [ex.submit(oracle_layer_cycle, orc, geom, st, cy, (done + i) % sample_layers, active, keep)
                    for i in range(cores)]
            for f in futs:
                f.result()
            done += cores
            el = time.perf_counter() - t0
            if el >= seconds or (max_layer_cycles and done >= max_layer_cycles):
                break
    el = time.perf_counter() - t0
    per_layer = el / done
    cycle_s = per_layer * n_layers
    return {"value": geom.B * geom.T / cycle_s, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": (f"{done} layer-cycles (verify+commit of one layer, B={geom.B} T={geom.T}) in "
                       f"{el:.1f} s on {cores} threads; scaled to a {n_layers}-layer cycle"),
            "seconds_per_cycle": cycle_s}


# ---------------------------------------------------------------- GPU arm
def timing_event():
    """A timing event that records as a graph node when captured."""
    import torch
    return torch.cuda.Event(enable_timing=True, external=True)


def verify_mode(mode, layer):
    """Layers after the first follow another layer's verify, which writes none of
    their buffers, so they may stage state (and in DEFERRED mode apply their
    pending commit) before that verify finishes.  Layer 0 follows the commit,
    which writes every layer's state or workspace."""
    from speculative_decode_gated_gdn_gb300 import lib as L
    return mode | (L.GDN_VERIFY_OVERLAP if layer > 0 else 0)


def run_gpu(args, rank, world, local):
    import torch
    from speculative_decode_gated_gdn_gb300 import lib as L
    from speculative_decode_gated_gdn_gb300 import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    geom, inactive = workload(args)
    n_layers = args.layers
    mode = MODES[args.mode]
    seed = rank_seed(args.seed, rank)
    pool = 16
    d = L.dims_of(geom)
    K, W = args.steps, args.warmup

    # persistent stack + input pool, all resident in HBM before timing
    st = synth.layer_state(geom, seed, n_layers)
    active_np = synth.active_mask(geom.B, inactive)
    keeps_np = synth.keep_draws(geom, seed, K + W)
    inp = [synth.cycle_inputs(geom, seed, p, n_layers) for p in range(pool)]
    if args.accept:
        # synthetic logits per pool entry, and per cycle drafts that repeat the
        # targets for the drawn number of positions: greedy acceptance then
        # reproduces the draw (at least 1: position 0 is always kept)
        V = args.V
        lg_bits = [synth.normal_bf16(seed + 7, f"logits{p}", geom.B * geom.T * V).reshape(geom.B, geom.T, V)
                   for p in range(pool)]
        tg = [np.argmax(synth.bf16_to_f32(bb), axis=2) for bb in lg_bits]
        keeps_np = np.maximum(keeps_np, 1).astype(np.int32)
        drafts_np = np.zeros((K + W, geom.B, geom.T), np.int32)
        for c in range(K + W):
            t_p = tg[c % pool]
            for b in range(geom.B):
                k = int(keeps_np[c, b])
                drafts_np[c, b, 1:k] = t_p[b, :k - 1]
                if k < geom.T:
                    drafts_np[c, b, k] = (t_p[b, k - 1] + 1) % V

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    state = torch.from_numpy(st["state"]).to(dev)
    ring = bf(st["ring"])
    conv_w = bf(st["conv_w"])
    offsets = torch.from_numpy(st["offsets"].copy()).to(dev)
    active = torch.from_numpy(active_np).to(dev)
    keeps = torch.from_numpy(keeps_np).to(dev)
    ws_bytes = L.gdn_layer_workspace_bytes(d, mode)
    ws = [torch.zeros(ws_bytes, dtype=torch.uint8, device=dev) for _ in range(n_layers)]  # DEFERRED: zeroed
    out = torch.empty((n_layers, geom.B, geom.T, geom.H_v, geom.d), dtype=torch.bfloat16, device=dev)
    xs = [bf(c["x"]) for c in inp]
    gs = [torch.from_numpy(c["g"]).to(dev) for c in inp]
    bs = [torch.from_numpy(c["beta"]).to(dev) for c in inp]
    states = [state[l] for l in range(n_layers)]
    rings = [ring[l] for l in range(n_layers)]
    if args.gated:
        zs = [bf(synth.normal_bf16(seed + 11, f"gate{p}", geom.B * geom.T * geom.H_v * geom.d)) for p in range(pool)]
        norm_w = bf(synth.normal_bf16(seed, "norm_w", geom.d, std=0.5))
    if args.accept:
        lgs = [bf(bb) for bb in lg_bits]
        drafts = torch.from_numpy(drafts_np).to(dev)
        keep_dev = torch.zeros(geom.B, dtype=torch.int32, device=dev)
        next_dev = torch.zeros(geom.B, dtype=torch.int32, device=dev)
        ws_acc = torch.zeros(L.gdn_accept_workspace_bytes(geom.B, geom.T, args.V), dtype=torch.uint8, device=dev)

    def cycle(c, x, g, beta, keep, ev=None):
        for l in range(n_layers):
            if args.gated:
                L.gdn_conv_verify_gated(d, verify_mode(mode, l), x[l], conv_w[l], g[l], beta[l], state[l], ring[l],
                                        offsets, active, zs[c % pool].view(geom.B, geom.T, geom.H_v, geom.d), norm_w,
                                        1e-6, out[l], ws[l], ws_bytes)
            else:
                L.gdn_conv_verify(d, verify_mode(mode, l), x[l], conv_w[l], g[l], beta[l], state[l], ring[l],
                                  offsets, active, out[l], ws[l], ws_bytes)
        if args.accept:
            L.gdn_accept_greedy(lgs[c % pool], drafts[c], active, keep_dev, next_dev, ws_acc)
            keep = keep_dev
        if ev is not None:
            ev[0].record()
        L.gdn_commit(d, mode, states, rings, ws, keep, active, offsets)
        if ev is not None:
            ev[1].record()

    # one CUDA graph per cycle (distinct keep row and timing events per cycle)
    side = torch.cuda.Stream(device=dev)
    graphs, events = [], []
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        cycle(0, xs[0], gs[0], bs[0], keeps[0])  # first calls outside capture
    torch.cuda.synchronize()
    for c in range(K + W):
        p = c % pool
        ev = (timing_event(), timing_event())
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=side):
            cycle(c, xs[p], gs[p], bs[p], keeps[c], ev)
        graphs.append(gr)
        events.append(ev)
    # restore the starting point the capture run disturbed
    state.copy_(torch.from_numpy(st["state"]).to(dev))
    ring.copy_(bf(st["ring"]))
    offsets.copy_(torch.from_numpy(st["offsets"].copy()).to(dev))
    for w in ws:
        w.zero_()
    torch.cuda.synchronize()

    for c in range(W):
        graphs[c].replay()
    torch.cuda.synchronize()

    import torch.distributed as dist
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    dev_id = f"GPU-{uuid}" if uuid is not None else str(local)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev_id) as clk:
        clk.mark_start()
        start.record()
        for c in range(W, W + K):
            graphs[c].replay()
        end.record()
        torch.cuda.synchronize()
        clk.mark_end()
    if world > 1:
        dist.barrier()
    ms = max_over_ranks(start.elapsed_time(end), dev, world)
    commit_ms = [events[c][0].elapsed_time(events[c][1]) for c in range(W, W + K)]

    n_active = int(active_np.sum())
    kp_all = np.where(active_np[None, :] == 1, keeps_np, 0)
    n_keep_all = (kp_all >= 1).sum(axis=1)
    n_keep = n_keep_all[W:W + K]
    # DEFERRED: the verify of cycle c applies the commit of cycle c - 1
    prev_keep = np.concatenate([[0], n_keep_all])  # [c] = kept rows of cycle c - 1 (none before cycle 0)
    n_apply = prev_keep[W:W + K] if args.mode == "deferred" else np.zeros(K, np.int64)
    commit_alg = np.array([commit_bytes(geom, int(nk), n_layers, args.mode) for nk in n_keep], dtype=np.float64)
    verify_alg = np.array([verify_bytes(geom, n_active, args.mode, int(na)) for na in n_apply], dtype=np.float64)
    step_bytes = commit_alg + n_layers * verify_alg
    min_bytes = np.array([path_min_bytes(geom, n_active, int(nk), n_layers) for nk in n_keep], dtype=np.float64)
    peak, peak_kind = measured_peak()
    step_ms = ms / K
    commit_avg_ms = float(np.mean(commit_ms))
    verify_avg_ms = max(step_ms - commit_avg_ms, 1e-9) / n_layers
    commit_gbs = float(commit_alg.mean()) / (commit_avg_ms * 1e-3) / 1e9
    verify_gbs = float(verify_alg.mean()) / (verify_avg_ms * 1e-3) / 1e9
    step_gbs = float(step_bytes.mean()) / (step_ms * 1e-3) / 1e9
    dominant = "commit" if commit_avg_ms >= verify_avg_ms * n_layers else "verify"
    wl_key = f"B{geom.B}T{geom.T}L{n_layers}{args.mode}"
    if dominant == "commit":
        roof = {"kernel": "commit_kernel (grouped over layers)", "bound": "hbm", "achieved": round(commit_gbs, 1),
                "peak": peak, "unit": "GB/s", "frac": round(commit_gbs / peak, 4),
                "traffic": profiled_traffic("commit", wl_key), "peak_source": peak_kind,
                "algorithmic_bytes_per_launch": float(commit_alg.mean()),
                "avg_launch_ms": round(commit_avg_ms, 5)}
    else:
        roof = {"kernel": "verify_kernel", "bound": "hbm", "achieved": round(verify_gbs, 1), "peak": peak,
                "unit": "GB/s", "frac": round(verify_gbs / peak, 4),
                "traffic": profiled_traffic("verify", wl_key), "peak_source": peak_kind,
                "algorithmic_bytes_per_launch": float(verify_alg.mean()),
                "avg_launch_ms": round(verify_avg_ms, 5)}
    res = {
        "metric": METRIC, "value": job_rate(world, geom.B * geom.T, step_ms), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": config_dict(args, geom, inactive),
        "hbm": {"step_algorithmic_bytes": float(step_bytes.mean()), "achieved_gbs": round(step_gbs, 1),
                "peak_gbs": peak, "frac": round(step_gbs / peak, 4), "peak_source": peak_kind,
                "path_min_bytes": float(min_bytes.mean()),
                "path_min_frac": round(float(min_bytes.mean()) / (step_ms * 1e-3) / 1e9 / peak, 4),
                "verify_gbs": round(verify_gbs, 1), "verify_avg_ms_incl_gaps": round(verify_avg_ms, 5),
                "commit_gbs": round(commit_gbs, 1), "commit_avg_ms": round(commit_avg_ms, 5)},
        "roofline": roof,
        "gpu_launches": K * (n_layers + 1 + int(args.accept)),
        "clocks": clk.summary(),
    }

    # end to end through the C ABI with host buffers: pinned inputs copied in,
    # outputs and offsets copied out, every step
    if not args.no_e2e:
        res["e2e"] = run_e2e(args, geom, d, mode, dev, inp, keeps_np, state, ring, conv_w, offsets, active,
                             ws, ws_bytes, out, states, world)
    del graphs
    return res


def run_e2e(args, geom, d, mode, dev, inp, keeps_np, state, ring, conv_w, offsets, active, ws, ws_bytes, out,
            states, world):
    import torch
    from speculative_decode_gated_gdn_gb300 import lib as L
    n_layers = args.layers
    K, W = args.steps, args.warmup
    pool = len(inp)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    hx = [pin(c["x"].view(np.int16)) for c in inp]
    hg = [pin(c["g"]) for c in inp]
    hb = [pin(c["beta"]) for c in inp]
    hk = pin(keeps_np)
    hout = torch.empty(out.shape, dtype=torch.bfloat16).pin_memory()
    hoff = torch.empty(offsets.shape, dtype=torch.int32).pin_memory()
    dx = torch.empty(hx[0].shape, dtype=torch.int16, device=dev)
    dg = torch.empty(hg[0].shape, dtype=torch.float32, device=dev)
    db = torch.empty(hb[0].shape, dtype=torch.float32, device=dev)
    dk = torch.empty((geom.B,), dtype=torch.int32, device=dev)
    dxb = dx.view(torch.bfloat16)

    def step(c):
        p = c % pool
        dx.copy_(hx[p], non_blocking=True)
        dg.copy_(hg[p], non_blocking=True)
        db.copy_(hb[p], non_blocking=True)
        dk.copy_(hk[c], non_blocking=True)
        for l in range(n_layers):
            L.gdn_conv_verify(d, verify_mode(mode, l), dxb[l], conv_w[l], dg[l], db[l], state[l], ring[l],
                              offsets, active, out[l], ws[l], ws_bytes)
        L.gdn_commit(d, mode, states, [ring[l] for l in range(n_layers)], ws, dk, active, offsets)
        hout.copy_(out, non_blocking=True)
        hoff.copy_(offsets, non_blocking=True)

    side = torch.cuda.Stream(device=dev)
    graphs = []
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        step(0)
    torch.cuda.synchronize()
    for c in range(K + W):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=side):
            step(c)
        graphs.append(gr)
    for c in range(W):
        graphs[c].replay()
    torch.cuda.synchronize()
    import torch.distributed as dist
    if world > 1:
        dist.barrier()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for c in range(W, W + K):
        graphs[c].replay()
    end.record()
    torch.cuda.synchronize()
    ms = max_over_ranks(start.elapsed_time(end), dev, world)
    h2d = hx[0].numel() * 2 + hg[0].numel() * 4 + hb[0].numel() * 4 + geom.B * 4
    d2h = hout.numel() * 2 + hoff.numel() * 4
    return {"value": job_rate(world, geom.B * geom.T, ms / K), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms / K,
            "how": "per step: pinned-host x/g/beta/keep copied in, 30 verifies + grouped commit through the C ABI, "
                   "outputs and offsets copied out; one CUDA graph per step"}


# ---------------------------------------------------------------- prefill leg
def prefill_flops(L, H_v, d, chunk=64):
    """Algorithmic FLOPs of the chunked form per prompt: per (chunk, value head)
    K K^T, Q K^T, W, U (n x n x d each), E = U - W S^T, Q S^T, S += K~^T E
    (n x d x d each), Pm E (n x n x d), plus the n^3/3 triangular solve."""
    total = 0
    for c0 in range(0, L, chunk):
        n = min(chunk, L - c0)
        total += H_v * (4 * 2 * n * n * d + 3 * 2 * n * d * d + 2 * n * n * d + n ** 3 // 3)
    return total


def run_accept_bench(args, rank, world, local):
    """Time gdn_accept_greedy alone: B x T positions over a V-entry vocabulary
    per launch, logits rotated over more distinct buffers than L2 holds."""
    import torch
    from speculative_decode_gated_gdn_gb300 import lib as L
    from speculative_decode_gated_gdn_gb300 import synth
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B, T, V, K, W = args.B, args.T, args.V, args.steps, args.warmup
    seed = rank_seed(args.seed, rank)
    base = [synth.normal_bf16(seed, f"logits{i}", B * T * V).reshape(B, T, V) for i in range(4)]
    per = B * T * V * 2
    n_buf = max(8, int(3 * 129e6 // per) + 1)  # three times L2 between reuses
    lgs = [torch.from_numpy(base[i % 4].view(np.int16)).to(dev).view(torch.bfloat16) for i in range(n_buf)]
    draft = torch.zeros((B, T), dtype=torch.int32, device=dev)
    active = torch.from_numpy(synth.active_mask(B, workload(args)[1])).to(dev)
    keep = torch.zeros(B, dtype=torch.int32, device=dev)
    nxt = torch.zeros(B, dtype=torch.int32, device=dev)
    ws = torch.zeros(L.gdn_accept_workspace_bytes(B, T, V), dtype=torch.uint8, device=dev)
    # K launches in one CUDA graph, so the device time is measured, not the
    # host's launch rate
    side = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(side):
        for i in range(W):
            L.gdn_accept_greedy(lgs[i % n_buf], draft, active, keep, nxt, ws)
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=side):
        for i in range(K):
            L.gdn_accept_greedy(lgs[i % n_buf], draft, active, keep, nxt, ws)
    gr.replay()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    gr.replay()
    end.record()
    torch.cuda.synchronize()
    ms = max_over_ranks(start.elapsed_time(end), dev, world) / K
    n_active = int(active.sum().item())
    alg = n_active * T * V * 2
    peak, peak_kind = measured_peak()
    gbs = alg / (ms * 1e-3) / 1e9
    return {"metric": "greedy acceptance positions/s", "value": job_rate(world, B * T, ms), "unit": "positions/s",
            "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"gdn_accept_greedy B={B} T={T} V={V}, {n_active} active rows, "
                                   f"{n_buf} logits buffers in rotation", "B": B, "T": T, "V": V},
            "roofline": {"kernel": "accept_kernel", "bound": "hbm", "achieved": round(gbs, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(gbs / peak, 4), "traffic": None, "peak_source": peak_kind,
                         "algorithmic_bytes_per_launch": alg, "avg_launch_ms": round(ms, 5)},
            "gpu_launches": K}


def run_prefill_bench(args, rank, world, local):
    """Time gdn_prefill_chunked: B rows primed over L tokens per step."""
    import torch
    from speculative_decode_gated_gdn_gb300 import lib as L
    from speculative_decode_gated_gdn_gb300 import synth
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    geom = synth.Geometry(B=args.B if args.B != 8 else 1, T=2, H_k=16, H_v=32, d=128)
    Lp, K, W = args.L, args.steps, args.warmup
    d = L.dims_of(geom)
    pr = synth.prompt_inputs(geom, rank_seed(args.seed, rank), Lp)
    st = synth.layer_state(geom, rank_seed(args.seed, rank), 1, offsets=np.zeros(geom.B, np.int32))

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    x, w = bf(pr["x"]), bf(st["conv_w"][0])
    g, beta = torch.from_numpy(pr["g"]).to(dev), torch.from_numpy(pr["beta"]).to(dev)
    state = torch.zeros((geom.B, geom.H_v, geom.d, geom.d), dtype=torch.float32, device=dev)
    ring = torch.zeros((geom.B, geom.R, geom.C), dtype=torch.bfloat16, device=dev)
    offsets = torch.zeros(geom.B, dtype=torch.int32, device=dev)
    out = torch.empty((geom.B, Lp, geom.H_v, geom.d), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(L.gdn_prefill_workspace_bytes(d, Lp), dtype=torch.uint8, device=dev)

    def step():
        L.gdn_prefill_chunked(d, Lp, x, w, g, beta, state, ring, offsets, out, ws)

    for _ in range(W):
        step()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(K):
        step()
    end.record()
    torch.cuda.synchronize()
    ms = max_over_ranks(start.elapsed_time(end), dev, world) / K
    flops = prefill_flops(Lp, geom.H_v, geom.d) * geom.B
    hbm = geom.B * (Lp * geom.C * 2 + Lp * geom.H_v * geom.d * 2 + 2 * geom.H_v * geom.d * geom.d * 4
                    + 2 * Lp * geom.H_v * 4)
    return {"metric": "GDN chunked prefill prompt tokens/s", "value": job_rate(world, geom.B * Lp, ms),
            "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": ms,
            "higher_is_better": True, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"chunked prefill B={geom.B} L={Lp} H_k=16 H_v=32 d=128 chunk 64",
                       "B": geom.B, "L": Lp},
            "algorithmic_gflop_per_step": flops / 1e9, "achieved_tflops": flops / (ms * 1e-3) / 1e12,
            "algorithmic_hbm_mb_per_step": hbm / 1e6, "achieved_hbm_gbs": hbm / (ms * 1e-3) / 1e9}


# ---------------------------------------------------------------- reference arm
def run_reference(args, rank, world):
    """The oracle (plain fp64 C, as it stands) on the host cores, on this
    arm's workload and metric; each step is a bounded sample of a cycle."""
    if rank != 0:
        return None
    geom, inactive = workload(args)
    K, W = args.steps, args.warmup
    import oracle
    from speculative_decode_gated_gdn_gb300 import synth
    orc = oracle.default()
    n_layers = args.layers
    sample_layers = min(n_layers, 4)
    st = synth.layer_state(geom, args.seed, sample_layers)
    cy = synth.cycle_inputs(geom, args.seed, 0, sample_layers)
    active = synth.active_mask(geom.B, inactive)
    cores = os.cpu_count() or 1
    budget_s = 150.0
    t0 = time.perf_counter()
    oracle_layer_cycle(orc, geom, st, cy, 0, active, cy["keep"])
    t_layer = time.perf_counter() - t0
    per_step_budget = budget_s / max(K + W, 1)
    # layers per step: one wave of threads at least, no more than the cycle, within budget
    waves = max(1, int(per_step_budget / max(t_layer, 1e-6)))
    per_step = max(1, min(n_layers, waves * cores))
    keeps = synth.keep_draws(geom, args.seed, K + W)
    times = []
    with concurrent.futures.ThreadPoolExecutor(max_workers=cores) as ex:
        for c in range(K + W):
            s0 = time.perf_counter()
            futs = [ex.submit(oracle_layer_cycle, orc, geom, st, cy, i % sample_layers, active, keeps[c])
                    for i in range(per_step)]
            for f in futs:
                f.result()
            if c >= W:
                times.append(time.perf_counter() - s0)
    step_s = float(np.mean(times)) * n_layers / per_step
    value = geom.B * geom.T / step_s
    sample = (f"each step: verify+commit of {per_step} of the {n_layers} layers (B={geom.B}, T={geom.T}, "
              f"full heads) on {cores} threads, scaled to the {n_layers}-layer cycle")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config_dict(args, geom, inactive),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse_args()
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend=backend)
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if args.workload in ("prefill", "accept"):
        res = (run_prefill_bench if args.workload == "prefill" else run_accept_bench)(args, rank, world, local)
        if rank == 0:
            print(json.dumps(res), flush=True)
        return
    res = run_gpu(args, rank, world, local)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            geom, inactive = workload(args)
            res["cpu_baseline"] = run_oracle_sample(geom, inactive, args.layers, args.cpu_seconds)
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
