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
The C-ABI calls of 64 consecutive cycles are captured in one CUDA graph, so
every kernel follows its predecessor with programmatic dependent launch, across
cycle boundaries too; the timed region is the replay of those graphs, with no
event inside it.  The verify's share of a cycle is measured as a marginal cost:
the same cycles are timed over half the stack, and a layer costs the
difference per layer.  Beside the headline the default run also times the
batch/draft sweep (B8/T8, B64/T2, B64/T8) and the chunked prefill of one row
at L = 4096 and 32768 (--no-extras skips them).

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
    "verify": ["speculative_decode_gated_gdn_gb300/csrc/verify_tc.cuh",
               "speculative_decode_gated_gdn_gb300/csrc/gdn_common.cuh"],
    "prefill": ["speculative_decode_gated_gdn_gb300/csrc/prefill.cu",
                "speculative_decode_gated_gdn_gb300/csrc/gdn_common.cuh"],
}


MODES = {"recompute": 0, "snapshot": 1, "deferred": 2}  # GDN_COMMIT_* of the C ABI


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=512)
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
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the batch/draft sweep and the prefill records beside the headline")
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


def code_only(src):
    """C/C++/CUDA source without its comments, trailing blanks and empty lines
    (string and character literals kept as written), so that a hash of it
    follows the code and not its commentary."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return "\n".join(line.rstrip() for line in "".join(out).splitlines() if line.strip())


def source_hash(kind):
    """Hash of the code (comments excluded) of the sources a profile entry covers."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(code_only(f.read()).encode())
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


def run_oracle_sample(geom, inactive, n_layers, seconds, max_layer_cycles=None, seed=2, cores=None):
    """Time the oracle on a bounded sample of layer-cycles using `cores` host
    threads (all host cores by default; threads over independent layers, the C
    oracle runs without the GIL)."""
    import oracle
    from speculative_decode_gated_gdn_gb300 import synth
    orc = oracle.default()
    sample_layers = min(n_layers, 4)
    st = synth.layer_state(geom, seed, sample_layers)
    cy = synth.cycle_inputs(geom, seed, 0, sample_layers)
    active = synth.active_mask(geom.B, inactive)
    keep = cy["keep"]
    cores = cores or os.cpu_count() or 1
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
CHUNK = 64  # cycles per captured graph (a graph of a few thousand kernel nodes)


def verify_mode(mode, layer):
    """Layers after the first follow another layer's verify, which writes none of
    their buffers, so they may stage state (and in DEFERRED mode apply their
    pending commit) before that verify finishes.  Layer 0 follows the commit:
    a DEFERRED commit writes no state, taps or captures, so layer 0 may still
    stage those early (GDN_VERIFY_OVERLAP_STATE); an eager commit writes the
    state, so layer 0 waits."""
    from speculative_decode_gated_gdn_gb300 import lib as L
    if layer > 0:
        return mode | L.GDN_VERIFY_OVERLAP
    return mode | (L.GDN_VERIFY_OVERLAP_STATE if mode == L.GDN_COMMIT_DEFERRED else 0)


class Stack:
    """Device tensors of one benchmark cohort (n-layer state stack, input pool)
    and the captured verify+commit cycles."""

    def __init__(self, args, geom, inactive, n_layers, seed, dev, pool=16, keep_cycles=0):
        import torch
        from speculative_decode_gated_gdn_gb300 import lib as L
        from speculative_decode_gated_gdn_gb300 import synth
        self.L, self.torch, self.args, self.geom, self.n_layers, self.dev = L, torch, args, geom, n_layers, dev
        self.mode = MODES[args.mode]
        self.pool = pool
        self.d = L.dims_of(geom)
        # the seeded draws of synth, made on the device (the host generator
        # would take minutes for the larger cohorts)
        st = synth.layer_state_dev(geom, seed, n_layers, dev)
        self.st0 = {k: v.clone() for k, v in st.items()}  # the starting point, for restore()
        self.active_np = synth.active_mask(geom.B, inactive)
        self.keeps_np = synth.keep_draws(geom, seed, keep_cycles)
        inp = [synth.cycle_inputs_dev(geom, seed, p, n_layers, dev) for p in range(pool)]
        self.state, self.ring, self.conv_w, self.offsets = st["state"], st["ring"], st["conv_w"], st["offsets"]
        self.active = torch.from_numpy(self.active_np).to(dev)
        self.keeps = torch.from_numpy(self.keeps_np).to(dev)
        self.ws_bytes = L.gdn_layer_workspace_bytes(self.d, self.mode)
        self.ws = [torch.zeros(self.ws_bytes, dtype=torch.uint8, device=dev) for _ in range(n_layers)]
        self.out = torch.empty((n_layers, geom.B, geom.T, geom.H_v, geom.d), dtype=torch.bfloat16, device=dev)
        self.xs = [c["x"] for c in inp]
        self.gs = [c["g"] for c in inp]
        self.bs = [c["beta"] for c in inp]
        self.side = torch.cuda.Stream(device=dev)
        self.extras = {}

    def bf(self, bits):
        t = self.torch
        return t.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(self.dev).view(t.bfloat16)

    def restore(self):
        """The starting point of a run: initial state, rings, offsets, zeroed workspaces."""
        self.state.copy_(self.st0["state"])
        self.ring.copy_(self.st0["ring"])
        self.offsets.copy_(self.st0["offsets"])
        for w in self.ws:
            w.zero_()

    def cycle(self, c, n_lay=None, x=None, g=None, beta=None, keep=None, out=None, hooks=None):
        """One verify+commit cycle over the first n_lay layers, issued on the
        current stream (captured into a graph by the caller); hooks[l] (if
        given) runs just before layer l's verify is issued."""
        L, a = self.L, self.args
        n = self.n_layers if n_lay is None else n_lay
        p = c % self.pool
        x = self.xs[p] if x is None else x
        g = self.gs[p] if g is None else g
        beta = self.bs[p] if beta is None else beta
        keep = self.keeps[c] if keep is None else keep
        out = self.out if out is None else out
        for l in range(n):
            if hooks and l in hooks:
                hooks[l]()
            if a.gated:
                L.gdn_conv_verify_gated(self.d, verify_mode(self.mode, l), x[l], self.conv_w[l], g[l], beta[l],
                                        self.state[l], self.ring[l], self.offsets, self.active,
                                        self.extras["zs"][p].view(self.geom.B, self.geom.T, self.geom.H_v,
                                                                  self.geom.d),
                                        self.extras["norm_w"], 1e-6, out[l], self.ws[l], self.ws_bytes)
            else:
                L.gdn_conv_verify(self.d, verify_mode(self.mode, l), x[l], self.conv_w[l], g[l], beta[l],
                                  self.state[l], self.ring[l], self.offsets, self.active, out[l], self.ws[l],
                                  self.ws_bytes)
        if a.accept:
            e = self.extras
            L.gdn_accept_greedy(e["lgs"][p], e["drafts"][c], self.active, e["keep_dev"], e["next_dev"], e["ws_acc"])
            keep = e["keep_dev"]
        L.gdn_commit(self.d, self.mode, [self.state[l] for l in range(n)], [self.ring[l] for l in range(n)],
                     self.ws[:n], keep, self.active, self.offsets)

    def capture(self, cycles, n_lay=None):
        """Graphs of up to CHUNK consecutive cycles each: every kernel of a chunk
        follows the previous one with programmatic dependent launch, across the
        cycle boundaries too."""
        torch = self.torch
        graphs = []
        for c0 in range(0, len(cycles), CHUNK):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=self.side):
                for c in cycles[c0:c0 + CHUNK]:
                    self.cycle(c, n_lay)
            graphs.append(gr)
        return graphs

    def time_graphs(self, warm, timed, clocks=None):
        """Replay the warm-up graphs, then time the others with CUDA events on
        the replay stream (synchronised on both sides); milliseconds."""
        torch = self.torch
        self.restore()
        torch.cuda.synchronize()
        for g in warm:
            g.replay()
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if clocks:
            clocks.mark_start()
        start.record()
        for g in timed:
            g.replay()
        end.record()
        torch.cuda.synchronize()
        if clocks:
            clocks.mark_end()
        return start.elapsed_time(end)


def cycle_bytes(geom, mode, active_np, keeps_np, W, K, n_layers):
    """Per-cycle algorithmic bytes of the timed cycles W..W+K-1 (verify, commit,
    whole step) and the path minimum, from the cycles' actual keep[] and active[]."""
    n_active = int(active_np.sum())
    kp_all = np.where(active_np[None, :] == 1, keeps_np, 0)
    n_keep_all = (kp_all >= 1).sum(axis=1)
    n_keep = n_keep_all[W:W + K]
    prev_keep = np.concatenate([[0], n_keep_all])  # DEFERRED: the verify of cycle c applies cycle c-1's commit
    n_apply = prev_keep[W:W + K] if mode == "deferred" else np.zeros(K, np.int64)
    commit_alg = np.array([commit_bytes(geom, int(nk), n_layers, mode) for nk in n_keep], dtype=np.float64)
    verify_alg = np.array([verify_bytes(geom, n_active, mode, int(na)) for na in n_apply], dtype=np.float64)
    step = commit_alg + n_layers * verify_alg
    pmin = np.array([path_min_bytes(geom, n_active, int(nk), n_layers) for nk in n_keep], dtype=np.float64)
    return verify_alg.mean(), commit_alg.mean(), step.mean(), pmin.mean()


def measure_cycles(args, geom, inactive, n_layers, K, W, seed, dev, world=1, clocks=None, marginal=True):
    """Build a cohort, capture W warm-up and K timed cycles in chained graphs
    and time them; with `marginal`, also time K2 cycles of the first half of
    the stack, so that a layer's cost is the difference per layer and the
    commit's the rest.  Returns (Stack, dict of times and bytes)."""
    import torch
    import torch.distributed as dist
    from speculative_decode_gated_gdn_gb300 import synth
    sk = Stack(args, geom, inactive, n_layers, seed, dev, keep_cycles=K + W)
    if args.accept:
        # synthetic logits per pool entry, and per cycle drafts that repeat the
        # targets for the drawn number of positions: greedy acceptance then
        # reproduces the draw (at least 1: position 0 is always kept)
        V = args.V
        lg_bits = [synth.normal_bf16(seed + 7, f"logits{p}", geom.B * geom.T * V).reshape(geom.B, geom.T, V)
                   for p in range(sk.pool)]
        tg = [np.argmax(synth.bf16_to_f32(bb), axis=2) for bb in lg_bits]
        sk.keeps_np = np.maximum(sk.keeps_np, 1).astype(np.int32)
        drafts_np = np.zeros((K + W, geom.B, geom.T), np.int32)
        for c in range(K + W):
            t_p = tg[c % sk.pool]
            for b in range(geom.B):
                k = int(sk.keeps_np[c, b])
                drafts_np[c, b, 1:k] = t_p[b, :k - 1]
                if k < geom.T:
                    drafts_np[c, b, k] = (t_p[b, k - 1] + 1) % V
        sk.extras.update(lgs=[sk.bf(bb) for bb in lg_bits], drafts=torch.from_numpy(drafts_np).to(dev),
                         keep_dev=torch.zeros(geom.B, dtype=torch.int32, device=dev),
                         next_dev=torch.zeros(geom.B, dtype=torch.int32, device=dev),
                         ws_acc=torch.zeros(sk.L.gdn_accept_workspace_bytes(geom.B, geom.T, V), dtype=torch.uint8,
                                            device=dev))
    if args.gated:
        sk.extras.update(zs=[sk.bf(synth.normal_bf16(seed + 11, f"gate{p}", geom.B * geom.T * geom.H_v * geom.d))
                             for p in range(sk.pool)],
                         norm_w=sk.bf(synth.normal_bf16(seed, "norm_w", geom.d, std=0.5)))
    # first calls outside capture (per-device library set-up), then the graphs
    torch.cuda.synchronize()
    with torch.cuda.stream(sk.side):
        sk.cycle(0)
    torch.cuda.synchronize()
    warm = sk.capture(list(range(W)))
    timed = sk.capture(list(range(W, W + K)))
    half = n_layers // 2
    K2 = min(K, 256)
    do_half = marginal and half >= 1 and not args.accept
    warm_h = sk.capture(list(range(W)), half) if do_half else None
    timed_h = sk.capture(list(range(W, W + K2)), half) if do_half else None
    if world > 1:
        dist.barrier()
    ms = sk.time_graphs(warm, timed, clocks)
    if world > 1:
        dist.barrier()
    ms = max_over_ranks(ms, dev, world)
    step_ms = ms / K
    if do_half:
        half_ms = sk.time_graphs(warm_h, timed_h) / K2
        verify_ms = max((step_ms - half_ms) / (n_layers - half), 1e-9)
        commit_ms = max(step_ms - n_layers * verify_ms, 0.0)
        split = f"marginal layer cost: (cycle at {n_layers} layers - cycle at {half}) / {n_layers - half}"
    else:
        verify_ms, commit_ms, split = step_ms / n_layers, 0.0, "cycle / layers (commit included)"
    verify_alg, commit_alg, step_alg, min_alg = cycle_bytes(geom, args.mode, sk.active_np, sk.keeps_np, W, K,
                                                             n_layers)
    del warm, timed, warm_h, timed_h
    return sk, {"step_ms": step_ms, "verify_ms": verify_ms, "commit_ms": commit_ms, "split": split,
                "verify_alg": verify_alg, "commit_alg": commit_alg, "step_alg": step_alg, "min_alg": min_alg}


def run_gpu(args, rank, world, local):
    import torch
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    geom, inactive = workload(args)
    n_layers = args.layers
    K, W = args.steps, args.warmup
    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    dev_id = f"GPU-{uuid}" if uuid is not None else str(local)
    with ClockSampler(dev_id) as clk:
        sk, m = measure_cycles(args, geom, inactive, n_layers, K, W, rank_seed(args.seed, rank), dev, world, clk)
    step_ms, verify_ms = m["step_ms"], m["verify_ms"]
    peak, peak_kind = measured_peak()
    verify_gbs = m["verify_alg"] / (verify_ms * 1e-3) / 1e9
    step_gbs = m["step_alg"] / (step_ms * 1e-3) / 1e9
    wl_key = f"B{geom.B}T{geom.T}L{n_layers}{args.mode}"
    res = {
        "metric": METRIC, "value": job_rate(world, geom.B * geom.T, step_ms), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": config_dict(args, geom, inactive),
        "hbm": {"step_algorithmic_bytes": m["step_alg"], "achieved_gbs": round(step_gbs, 1),
                "peak_gbs": peak, "frac": round(step_gbs / peak, 4), "peak_source": peak_kind,
                "path_min_bytes": m["min_alg"],
                "path_min_frac": round(m["min_alg"] / (step_ms * 1e-3) / 1e9 / peak, 4),
                "verify_gbs": round(verify_gbs, 1), "verify_ms": round(verify_ms, 5),
                "commit_ms": round(m["commit_ms"], 5), "split": m["split"]},
        "roofline": {"kernel": "verify_tc_kernel (d=128)" if geom.d == 128 and args.mode != "snapshot"
                     else "verify_kernel", "bound": "hbm", "achieved": round(verify_gbs, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(verify_gbs / peak, 4),
                     "traffic": profiled_traffic("verify", wl_key), "peak_source": peak_kind,
                     "algorithmic_bytes_per_launch": m["verify_alg"], "avg_launch_ms": round(verify_ms, 5),
                     "launch_duration": m["split"]},
        "gpu_launches": K * (n_layers + 1 + int(args.accept)),
        "clocks": clk.summary(),
    }
    if not args.no_e2e:
        res["e2e"] = run_e2e(args, sk, world)
    del sk
    torch.cuda.empty_cache()
    return res


SWEEP = [(8, 8), (64, 2), (64, 8)]  # (B, T) of the batch/draft sweep beside the headline


def run_sweep(args, dev):
    """The batch/draft sweep (30 layers, the last B/4 rows inactive, keep ~
    U{0..T}) at a few cohorts, each timed like the headline but shorter."""
    import copy
    import torch
    from speculative_decode_gated_gdn_gb300 import synth
    out = []
    peak, peak_kind = measured_peak()
    for B, T in SWEEP:
        a = copy.copy(args)
        a.B, a.T, a.gated, a.accept, a.inactive = B, T, False, False, None
        geom, inactive = workload(a)
        sk, m = measure_cycles(a, geom, inactive, a.layers, 64, 4, a.seed, dev)
        del sk
        torch.cuda.empty_cache()
        out.append({"B": B, "T": T, "layers": a.layers, "row_tokens_per_s": round(B * T / (m["step_ms"] * 1e-3), 1),
                    "ms_per_cycle": round(m["step_ms"], 5), "verify_us": round(m["verify_ms"] * 1e3, 3),
                    "verify_hbm_frac": round(m["verify_alg"] / (m["verify_ms"] * 1e-3) / 1e9 / peak, 4),
                    "path_min_frac": round(m["min_alg"] / (m["step_ms"] * 1e-3) / 1e9 / peak, 4),
                    "inactive_rows": list(inactive)})
    return {"cycles": 64, "mode": args.mode, "peak_gbs": peak, "peak_source": peak_kind, "entries": out}


def run_e2e(args, sk, world):
    """The same cycles through the C ABI with host buffers: every step copies its
    x/g/beta/keep in from pinned host memory and its outputs and offsets out,
    inside the timed region.  Inputs and outputs are double-buffered on the
    device and the copies run on a copy stream, ordered by events against the
    compute, so step c+1's copy-in and step c-1's copy-out overlap step c."""
    import torch
    geom, n_layers = sk.geom, sk.n_layers
    K, W = args.steps, args.warmup
    dev = sk.dev
    # every host buffer is a view of one pinned block (one allocation, 256-byte
    # aligned views): the copy engines see a few large translations instead of
    # many small pinned allocations scattered over host memory
    keeps_t = torch.from_numpy(np.ascontiguousarray(sk.keeps_np))
    srcs = ([x.view(torch.int16) for x in sk.xs] + list(sk.gs) + list(sk.bs) + [keeps_t]
            + [torch.empty(sk.out.shape, dtype=torch.bfloat16)] * 2 + [torch.empty(sk.offsets.shape, dtype=torch.int32)] * 2)
    sizes = [(t.numel() * t.element_size() + 255) // 256 * 256 for t in srcs]
    block = torch.empty(sum(sizes), dtype=torch.uint8, pin_memory=True)
    views, off = [], 0
    for t, n in zip(srcs, sizes):
        v = block[off:off + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
        v.copy_(t)  # the inputs' values (device tensors are copied to the host once here)
        views.append(v)
        off += n
    P = len(sk.xs)
    hx, hg, hb = views[:P], views[P:2 * P], views[2 * P:3 * P]
    hk = views[3 * P]
    hout, hoff = views[3 * P + 1:3 * P + 3], views[3 * P + 3:3 * P + 5]
    dx = [torch.empty(hx[0].shape, dtype=torch.int16, device=dev) for _ in range(2)]
    dg = [torch.empty(hg[0].shape, dtype=torch.float32, device=dev) for _ in range(2)]
    db = [torch.empty(hb[0].shape, dtype=torch.float32, device=dev) for _ in range(2)]
    dk = [torch.empty((geom.B,), dtype=torch.int32, device=dev) for _ in range(2)]
    dout = [torch.empty_like(sk.out) for _ in range(2)]
    doff = [torch.empty_like(sk.offsets) for _ in range(2)]
    h2d_s = torch.cuda.Stream(device=dev)  # copies in
    d2h_s = torch.cuda.Stream(device=dev)  # copies out

    def steps(cycles):
        """Steps of `cycles`, captured on sk.side (compute), h2d_s and d2h_s.

        Step c+1's copy-in is issued before step c's compute, and every wait
        the compute stream needs for step c+1 (its inputs in, the output
        buffer it reuses copied out, the offsets snapshot of step c-1 taken
        before step c+1's commit moves them) sits in the middle of step c's
        layer stack, where the copies are long done: only that one
        verify-to-verify edge per step loses its programmatic overlap, and
        only library kernels run on the compute stream."""
        ev_in = [torch.cuda.Event(), torch.cuda.Event()]
        ev_done = [torch.cuda.Event(), torch.cuda.Event()]
        ev_out = [torch.cuda.Event(), torch.cuda.Event()]
        ev_snap = [torch.cuda.Event(), torch.cuda.Event()]
        fresh = [True, True]
        h2d_s.wait_stream(sk.side)  # bring both copy streams into the capture
        d2h_s.wait_stream(sk.side)

        def copy_in(c):
            s, p = c % 2, c % sk.pool
            if not fresh[s]:
                h2d_s.wait_event(ev_done[s])  # step c-2's compute is done with buffer s
            with torch.cuda.stream(h2d_s):
                dx[s].copy_(hx[p], non_blocking=True)
                dg[s].copy_(hg[p], non_blocking=True)
                db[s].copy_(hb[p], non_blocking=True)
                dk[s].copy_(hk[c], non_blocking=True)
            ev_in[s].record(h2d_s)

        def waits_for(c):
            """What step c needs from the copy streams before it may run."""
            s = c % 2
            sk.side.wait_event(ev_in[s])
            if not fresh[s]:
                sk.side.wait_event(ev_out[s])   # step c-2's outputs are out of buffer s
                sk.side.wait_event(ev_snap[s])  # and its offsets snapshot is taken

        copy_in(cycles[0])
        waits_for(cycles[0])
        for i, c in enumerate(cycles):
            s = c % 2
            nxt = cycles[i + 1] if i + 1 < len(cycles) else None
            if nxt is not None:
                copy_in(nxt)
            hooks = {n_layers // 2: (lambda n=nxt: waits_for(n))} if nxt is not None else None
            with torch.cuda.stream(sk.side):
                sk.cycle(c, None, dx[s].view(torch.bfloat16), dg[s], db[s], dk[s], dout[s], hooks=hooks)
            ev_done[s].record(sk.side)
            # copy-out of step c: the offsets first (the next commit but one moves them), then the outputs
            d2h_s.wait_event(ev_done[s])
            with torch.cuda.stream(d2h_s):
                doff[s].copy_(sk.offsets)
                ev_snap[s].record(d2h_s)
                hout[s].copy_(dout[s], non_blocking=True)
                hoff[s].copy_(doff[s], non_blocking=True)
            ev_out[s].record(d2h_s)
            fresh[s] = False
        sk.side.wait_stream(h2d_s)  # join
        sk.side.wait_stream(d2h_s)

    graphs = []
    torch.cuda.synchronize()
    for cyc in ([list(range(W))] + [list(range(W + c0, min(W + K, W + c0 + CHUNK))) for c0 in range(0, K, CHUNK)]):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=sk.side):
            steps(cyc)
        graphs.append(gr)
    ms = sk.time_graphs(graphs[:1], graphs[1:])
    ms = max_over_ranks(ms, dev, world)
    h2d = hx[0].numel() * 2 + hg[0].numel() * 4 + hb[0].numel() * 4 + geom.B * 4
    d2h = hout[0].numel() * 2 + hoff[0].numel() * 4
    return {"value": job_rate(world, geom.B * geom.T, ms / K), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms / K,
            "how": "per step: pinned-host x/g/beta/keep copied in, 30 verifies + grouped commit through the C ABI, "
                   "outputs and offsets copied out; inputs/outputs double-buffered, copies on their own streams, "
                   "each step's waits on them placed mid-way through the previous step's layers so the copies "
                   "overlap compute and the chain keeps its overlap; CUDA graphs of 64 steps"}


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


def measure_prefill(L_prompt, K, W, seed, dev):
    """Time gdn_prefill_chunked priming one row (B = 1) over L_prompt tokens:
    milliseconds per call and the algorithmic work."""
    import torch
    from speculative_decode_gated_gdn_gb300 import lib as L
    from speculative_decode_gated_gdn_gb300 import synth
    geom = synth.Geometry(B=1, T=2, H_k=16, H_v=32, d=128)
    d = L.dims_of(geom)
    pr = synth.prompt_inputs(geom, seed, L_prompt)
    st = synth.layer_state(geom, seed, 1, offsets=np.zeros(geom.B, np.int32))

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    x, w = bf(pr["x"]), bf(st["conv_w"][0])
    g, beta = torch.from_numpy(pr["g"]).to(dev), torch.from_numpy(pr["beta"]).to(dev)
    state = torch.zeros((geom.B, geom.H_v, geom.d, geom.d), dtype=torch.float32, device=dev)
    ring = torch.zeros((geom.B, geom.R, geom.C), dtype=torch.bfloat16, device=dev)
    offsets = torch.zeros(geom.B, dtype=torch.int32, device=dev)
    out = torch.empty((geom.B, L_prompt, geom.H_v, geom.d), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(L.gdn_prefill_workspace_bytes(d, L_prompt), dtype=torch.uint8, device=dev)

    def step():
        L.gdn_prefill_chunked(d, L_prompt, x, w, g, beta, state, ring, offsets, out, ws)

    for _ in range(W):
        step()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(K):
        step()
    end.record()
    torch.cuda.synchronize()
    ms = start.elapsed_time(end) / K
    flops = prefill_flops(L_prompt, geom.H_v, geom.d) * geom.B
    hbm = geom.B * (L_prompt * geom.C * 2 + L_prompt * geom.H_v * geom.d * 2 + 2 * geom.H_v * geom.d * geom.d * 4
                    + 2 * L_prompt * geom.H_v * 4)
    del x, w, g, beta, state, ring, out, ws
    torch.cuda.empty_cache()
    return ms, flops, hbm, geom


def measured_tflops():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j["bf16_tflops_sustained"]), float(j["bf16_tflops"]), "measured"
    except Exception:
        return 1700.0, 1900.0, "fallback"


def prefill_record(args, dev):
    """Chunked prefill of one row at L = 4096 and 32768 (the state-priming
    configuration), with the tensor-pipe utilisation of its kernels from the
    committed ncu summary when that was taken on the current source."""
    sust, burst, kind = measured_tflops()
    entries = []
    for L_prompt, K, W in ((4096, 20, 3), (32768, 4, 1)):
        ms, flops, hbm, _ = measure_prefill(L_prompt, K, W, args.seed, dev)
        tf = flops / (ms * 1e-3) / 1e12
        entries.append({"L": L_prompt, "ms": round(ms, 4), "tokens_per_s": round(L_prompt / (ms * 1e-3), 1),
                        "algorithmic_gflop": round(flops / 1e9, 2), "achieved_tflops": round(tf, 2),
                        "frac_of_bf16_sustained": round(tf / sust, 4),
                        "hbm_gb_per_s": round(hbm / (ms * 1e-3) / 1e9, 1)})
    return {"B": 1, "chunk": 64, "peak_bf16_tflops_sustained": sust, "peak_source": kind,
            "tensor_pipe": profiled_tensor_pipe(), "entries": entries}


def profiled_tensor_pipe():
    """sm__pipe_tensor_cycles_active per prefill kernel from profiles/traffic.json,
    if taken on the current prefill source (null otherwise)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)["prefill"]
    except Exception:
        return None
    if rec.get("source_hash") != source_hash("prefill"):
        return None
    return rec.get("tensor_pipe")


def run_prefill_bench(args, rank, world, local):
    """Time gdn_prefill_chunked: B rows primed over L tokens per step."""
    import torch
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ms, flops, hbm, geom = measure_prefill(args.L, args.steps, args.warmup, rank_seed(args.seed, rank), dev)
    ms = max_over_ranks(ms, dev, world)
    sust, burst, kind = measured_tflops()
    tf = flops / (ms * 1e-3) / 1e12
    return {"metric": "GDN chunked prefill prompt tokens/s", "value": job_rate(world, geom.B * args.L, ms),
            "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"chunked prefill B={geom.B} L={args.L} H_k=16 H_v=32 d=128 chunk 64",
                       "B": geom.B, "L": args.L},
            "algorithmic_gflop_per_step": flops / 1e9, "achieved_tflops": tf,
            "frac_of_bf16_sustained": tf / sust, "peak_source": kind,
            "algorithmic_hbm_mb_per_step": hbm / 1e6, "achieved_hbm_gbs": hbm / (ms * 1e-3) / 1e9,
            "tensor_pipe": profiled_tensor_pipe()}


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
    if rank == 0 and world == 1 and not args.no_extras:
        import torch
        dev = torch.device("cuda", local)
        res["sweep"] = run_sweep(args, dev)
        res["prefill"] = prefill_record(args, dev)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            geom, inactive = workload(args)
            res["cpu_baseline"] = run_oracle_sample(geom, inactive, args.layers, args.cpu_seconds)
            one = run_oracle_sample(geom, inactive, args.layers, args.cpu_seconds / 3, cores=1)
            res["cpu_baseline"]["single_core"] = {k: one[k] for k in ("value", "unit", "cores", "sample",
                                                                      "seconds_per_cycle")}
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
