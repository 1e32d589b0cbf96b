"""Benchmark of the HiSparse RESOLVE hot path on one GB300 (or N replicas).

One *step* is one decode step of the whole hot path over every layer of the
workload: write-through of the previous token (backup stream), the new token's
KV placed in row B, RESOLVE on every anchor layer, and plan replay into every
shared-index layer.  Inputs for all steps are resident in HBM before timing.

Default workload: the DSA-style token-selection workload -- 8 requests x 4
layers, 128K context, k=2048, B=4096, 1152-byte records, one new token per
step written through.  Every rank (torchrun, one process per GPU) runs its own
replica of the workload (units are independent: weak scaling, no collective).

Printed (rank 0, one JSON line): selections/s over the whole job, the miss
fetch rate of the RESOLVE kernel against the host->device bandwidth measured
in the same run by a pinned cudaMemcpyAsync probe, the all-hit (no-IO) rate,
an end-to-end rate through the C ABI with host buffers, and the oracle timed
on the host cores.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "RESOLVE selections/s per layer-step; miss-fetch GB/s vs measured host-link peak"


# --------------------------------------------------------------------------- #
def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="dsa")
    ap.add_argument("--ctas", type=int, default=0, help="CTAs per request in resolve (0 = auto)")
    ap.add_argument("--replay-ctas", type=int, default=0)
    ap.add_argument("--lookup", type=int, default=0, help="0 = page table (default), 1 = hash")
    ap.add_argument("--pool", choices=["huge", "pinned"], default="pinned",
                    help="host pool kind: cudaHostAlloc (default) or huge-page registered")
    ap.add_argument("--no-burn-in", action="store_true",
                    help="skip the untimed passes over the trace before warm-up")
    ap.add_argument("--burn-in", type=int, default=3,
                    help="untimed passes over the trace before warm-up (default 3)")
    ap.add_argument("--resident", default="",
                    help="FULL,WINDOW,TOKENS: three-tier resolve with the first FULL requests "
                         "resident over their whole context and the others over their last "
                         "WINDOW positions, TOKENS positions per resident block")
    ap.add_argument("--verify-rows", type=int, default=1,
                    help="V > 1: each request's list is V speculative verify rows of top_k / V "
                         "selections, resolved as one union (HISPARSE_UNION)")
    ap.add_argument("--interleave", action="store_true",
                    help="host rows of each shared-index group (anchor + followers) "
                         "interleaved row by row, so replays read the pages the anchor's "
                         "fetch just read")
    ap.add_argument("--mirror", action="store_true",
                    help="fetch missed records from an HBM mirror of the host pool "
                         "(FROM_MIRROR): the same kernels with HBM as the source; the "
                         "roofline is then against HBM (write-backs store to both)")
    ap.add_argument("--unfused", action="store_true",
                    help="write-through as its own launch instead of inside RESOLVE")
    ap.add_argument("--L-ctx", type=int, default=0,
                    help="override the workload's prefill length (host pool size)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-copy", choices=("sm", "engine"), default="sm",
                    help="end-to-end pass: copy each step's inputs and results with SM "
                         "threads (hisparse_copy) or with the copy engines (cudaMemcpyAsync)")
    ap.add_argument("--replay", choices=("group", "layer", "inline"), default="group",
                    help="shared-index layers: one replay launch per anchor (group), one "
                         "per layer (layer, as the pages describe), or filled inside the "
                         "anchor's RESOLVE launch (inline, HISPARSE_WITH_SHARED)")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-allhit", action="store_true")
    ap.add_argument("--verify", dest="verify", action="store_true", default=True,
                    help="after the timed pass, compare its final state with the oracle "
                         "(the default)")
    ap.add_argument("--no-verify", dest="verify", action="store_false")
    ap.add_argument("--workloads", default=",".join(SUB_WORKLOADS),
                    help="the other workloads measured after the headline, each on its own "
                         "pool, reported in the line's `workloads` object (one GPU only)")
    ap.add_argument("--no-workloads", action="store_true")
    ap.add_argument("--skip-io", action="store_true",
                    help="every RESOLVE with SKIP_IO: the metadata path with the trace's "
                         "misses and no record copies (the pages' no-IO mode)")
    ap.add_argument("--no-alt-burn-in", action="store_true",
                    help="skip the timed pass after a burn-in over another trace")
    ap.add_argument("--l2-persist", type=int, default=0,
                    help="MB of L2 set aside to keep the RESOLVE layers' page tables "
                         "persisting between steps (hisparse_set_l2_persisting; 0 = off)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class Clocks:
    """Sample SM clocks and throttle reasons with nvidia-smi during a region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self._stop = threading.Event()
        self._th = None

    def _run(self):
        while not self._stop.is_set():
            try:
                out = subprocess.run(["nvidia-smi", "-i", str(self.index),
                                      f"--query-gpu={self.Q}", "--format=csv,noheader,nounits"],
                                     capture_output=True, text=True, timeout=5).stdout.strip()
                if out:
                    self.samples.append([x.strip() for x in out.split(",")])
            except Exception:
                pass
            self._stop.wait(0.2)

    def __enter__(self):
        self._th = threading.Thread(target=self._run, daemon=True)
        self._th.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        self._th.join(timeout=10)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(s[0]) for s in self.samples if s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in self.samples for i in range(4)
                          if len(s) > 4 + i and s[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.samples)}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            return json.load(fh), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def profile_traffic(kernel_file, kernel):
    """Per-launch traffic of `kernel` from the ncu summaries under profiles/.

    A summary line of the form
      machine: kernel=<name> sha256=<kernel source sha256> dram_bytes_per_launch=<n> sysmem_bytes_per_launch=<n> [algorithmic_bytes_per_launch=<n>]
    counts only while the kernel source still has that hash (the counters are
    stale once the kernel changes).  The captured launch's own miss bytes come
    with it: a launch's host-link traffic is in proportion to its misses, so the
    two are compared as a ratio.
    """
    sha = hashlib.sha256(open(kernel_file, "rb").read()).hexdigest()
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    for name in sorted(os.listdir(pdir)):
        if not name.endswith(".md"):
            continue
        for line in open(os.path.join(pdir, name), encoding="utf-8"):
            if not line.startswith("machine:"):
                continue
            kv = dict(x.split("=", 1) for x in line.split()[1:] if "=" in x)
            if kv.get("kernel") == kernel and kv.get("sha256") == sha:
                return {"dram_bytes_per_launch": float(kv["dram_bytes_per_launch"]),
                        "sysmem_bytes_per_launch": float(kv["sysmem_bytes_per_launch"]),
                        "algorithmic_bytes": (float(kv["algorithmic_bytes_per_launch"])
                                              if "algorithmic_bytes_per_launch" in kv else None),
                        "source": name}
    return None


# --------------------------------------------------------------------------- #
def token_traces(w, traces):
    """The traces as positions: block ids expanded for a block-selecting
    workload (block b -> positions b*t .. b*t + t - 1, -1 -> t paddings)."""
    import numpy as np
    t = w.sel_block_tokens
    if t <= 1:
        return traces
    out = {}
    for a, (blk, nw) in traces.items():
        pos = (blk[..., None].astype(np.int64) * t + np.arange(t)).reshape(*blk.shape[:-1], -1)
        out[a] = (np.where(np.repeat(blk == -1, t, axis=-1), -1, pos).astype(np.int32), nw)
    return out


def cpu_oracle_rate(w, traces, host_views=None, budget_s=10.0, union=False, warmup=0,
                    steps=None):
    """The C oracle (single thread) on the same workload's steps: selections/s.

    ``host_views[l]`` is a uint8 [R][>=L_ctx][rec] view of layer l's host rows
    (rows below L_ctx are read-only input); without it the rows are generated.
    With ``steps``, the first ``warmup`` steps run untimed and exactly the next
    ``steps`` are timed; otherwise steps from 0 are timed until the trace or
    ``budget_s`` ends.
    """
    import numpy as np
    from oracle.coracle import OracleLayer
    from workload import records as REC

    anchors = w.anchors()
    layers = {}
    for l in range(w.L):
        if host_views is not None:
            arr = host_views[l]
        else:
            arr = np.empty((w.R, w.L_ctx, w.rec), np.uint8)
            for r in range(w.R):
                REC.fill(arr[r].ctypes.data, w.L_ctx, w.rec, w.rec, w.seed, l, r, 0)
        layers[l] = OracleLayer(w.R, w.k, w.B, w.P, w.rec, host=arr, host_split=w.L_ctx,
                                metadata=l in anchors)
        if l in anchors:
            layers[l].reset()
            if w.admit_preload:   # short requests start admitted with their prefill
                for r in range(w.R):
                    layers[l].admit(r, w.L_ctx)
    new_rows = REC.new_token_records(w)
    anchor_of = w.anchor_of()
    sel_total, miss_bytes, steps_done, t_total = 0, 0, 0, 0.0
    t_start = time.perf_counter()
    t = 0
    timed_from = warmup if steps is not None else 0
    while True:
        if t == timed_from:
            sel_total, miss_bytes, steps_done, t_total = 0, 0, 0, 0.0
        t0 = time.perf_counter()
        if w.write_through:
            for l in range(w.L):
                if t > 0:
                    layers[l].writeback(traces[anchors[0]][1][t - 1])
                layers[l].set_newest_rows(new_rows[t, l])
        for a in anchors:
            nw = traces[a][1][t] if w.write_through else None
            if w.admit_preload:
                prev = traces[a][1][t - 1] if t > 0 else np.full(w.R, -1, np.int32)
                layers[a].resolve_with_seq_lens(traces[a][0][t], nw, prev,
                                                np.full(w.R, w.L_ctx + t + 1, np.int32))
            else:
                layers[a].resolve(traces[a][0][t], nw, union=union)
            miss_bytes += int(layers[a].miss_count.sum()) * w.rec
            for f in (l for l in range(w.L) if anchor_of[l] == a):
                layers[a].replay_into(layers[f])
        t_total += time.perf_counter() - t0
        sel_total += len(anchors) * w.R * w.k
        steps_done += 1
        t += 1
        if steps is not None:
            if t >= warmup + steps:
                break
        elif t >= w.steps or time.perf_counter() - t_start > budget_s:
            break
    which = (f"decode steps {timed_from}..{timed_from + steps_done - 1} (after {timed_from} "
             f"untimed)" if steps is not None else f"first {steps_done} decode steps")
    return {"value": sel_total / t_total, "unit": "selections/s", "cores": 1, "kind": "oracle",
            "sample": f"{which} of the {w.name} workload "
                      f"({w.R} requests x {w.L} layers, k={w.k}, B={w.B}), plain C oracle, "
                      f"one thread, record copies included, trace generation excluded",
            "miss_bytes_per_s": miss_bytes / t_total, "seconds": t_total,
            "steps": steps_done}


def cpu_oracle_rate_threads(w, traces, host_views, threads, union=False):
    """The same C oracle over all decode steps, with the workload's independent
    units -- one request of one anchor layer, with its shared-index layers --
    spread over `threads` Python threads (each oracle call releases the GIL)."""
    import numpy as np
    from concurrent.futures import ThreadPoolExecutor
    from oracle.coracle import OracleLayer
    from workload import records as REC

    anchors = w.anchors()
    anchor_of = w.anchor_of()
    new_rows = REC.new_token_records(w)
    units = []
    for a in anchors:
        fls = [l for l in range(w.L) if anchor_of[l] == a]
        for r in range(w.R):
            mk = lambda l, meta: OracleLayer(1, w.k, w.B, w.P, w.rec,
                                             host=host_views[l][r:r + 1], host_split=w.L_ctx,
                                             metadata=meta)
            units.append((a, r, mk(a, True), [(f, mk(f, False)) for f in fls]))
    for _, _, o, _ in units:
        o.reset()
        if w.admit_preload:
            o.admit(0, w.L_ctx)

    def run(chunk):
        sel = misses = 0
        for a, r, o, fls in chunk:
            for t in range(w.steps):
                if w.write_through:
                    for l, lay in [(a, o)] + fls:
                        if t > 0:
                            lay.writeback(traces[anchors[0]][1][t - 1][r:r + 1])
                        lay.set_newest_rows(new_rows[t, l, r:r + 1])
                nw = traces[a][1][t][r:r + 1] if w.write_through else None
                if w.admit_preload:
                    prev = traces[a][1][t - 1][r:r + 1] if t > 0 else np.full(1, -1, np.int32)
                    o.resolve_with_seq_lens(traces[a][0][t][r:r + 1], nw, prev,
                                            np.full(1, w.L_ctx + t + 1, np.int32))
                else:
                    o.resolve(traces[a][0][t][r:r + 1], nw, union=union)
                misses += int(o.miss_count.sum())
                for _, lay in fls:
                    o.replay_into(lay)
                sel += w.k
        return sel, misses

    chunks = [units[i::threads] for i in range(threads)]
    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        res = list(ex.map(run, chunks))
    dt = time.perf_counter() - t0
    sel = sum(x for x, _ in res)
    return {"value": sel / dt, "unit": "selections/s", "cores": threads, "kind": "oracle",
            "sample": f"all {w.steps} decode steps of the {w.name} workload, its "
                      f"{len(units)} independent (request, anchor layer) units spread over "
                      f"{threads} threads, plain C oracle, record copies included",
            "miss_bytes_per_s": sum(m for _, m in res) * w.rec / dt, "seconds": dt}


# --------------------------------------------------------------------------- #
TARGET_LINK_FRAC = 0.8   # the miss-fetch path's target share of the measured host link

# The default line's other workloads (name -> how it is built and run).
SUB_WORKLOADS = ("tiny", "quest", "short", "shared_inline", "shared_inline_huge",
                 "shared_anchor", "sweep", "sweep_huge", "sweep_allhit")
SWEEP_POINT = (4096, 0.87)           # (B, reuse fraction) of the capacity-sweep entry
SWEEP_CONTEXTS = (1048576, 524288, 262144)
HOST_MARGIN_GIB = 32                 # host memory left free beside a pinned pool


def opts_for(args, **kw):
    """A copy of the command-line options with some replaced."""
    d = dict(vars(args))
    d.update(kw)
    return argparse.Namespace(**d)


def workload_config(w, o, n_gpus):
    """The line's config: the workload and the options that shape the run (the
    same on both arms; facts of the run itself go elsewhere)."""
    return {"workload": w.name, "requests": w.R, "layers": w.L, "anchors": len(w.anchors()),
            "top_k": w.k, "B": w.B, "L_ctx": w.L_ctx, "record_bytes": w.rec,
            "write_through": w.write_through, "parallelism": f"replicas{n_gpus}",
            "l2": "flushed (256 MB write) before every timed step",
            "lookup": ["page_table", "hash"][o.lookup],
            "write_through_launch": "separate" if o.unfused else "fused into RESOLVE",
            "host_pool": o.pool,
            "replay_launch": {"group": "one per anchor for all its shared-index layers",
                              "layer": "one per shared-index layer",
                              "inline": "none: shared-index layers filled inside the "
                                        "anchor's RESOLVE"}[o.replay],
            "host_layout": ("rows of each shared-index group interleaved" if o.interleave
                            else "one block of rows per layer"),
            "fetch_source": "HBM mirror of the host pool" if o.mirror else "host pool",
            "verify_rows": o.verify_rows,
            "resident_tier": (dict(zip(("full_requests", "window", "tokens_per_block"),
                                       (int(x) for x in o.resident.split(","))))
                              if o.resident else None),
            "burn_in": None if o.no_burn_in else
            f"{o.burn_in} untimed passes over all steps, each from the admission state",
            "l2_persisting_mb": o.l2_persist or None}


def mem_available():
    """Host MemAvailable in bytes (0 if unknown)."""
    try:
        for line in open("/proc/meminfo"):
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def pick_sweep_context(B, f):
    """The largest capacity-sweep context whose pinned host pool leaves
    HOST_MARGIN_GIB of host memory free; every candidate and the outcome."""
    from workload import sweep_workload
    avail = mem_available()
    tried = []
    for L in SWEEP_CONTEXTS:
        need = sweep_workload(B, f, L_ctx=L).host_bytes()
        ok = avail >= need + (HOST_MARGIN_GIB << 30)
        tried.append({"L_ctx": L, "host_pool_gb": round(need / 1e9, 1), "fits": ok})
        if ok:
            return L, {"mem_available_gb": round(avail / 1e9, 1), "margin_gib": HOST_MARGIN_GIB,
                       "candidates": tried}
    return None, {"mem_available_gb": round(avail / 1e9, 1), "margin_gib": HOST_MARGIN_GIB,
                  "candidates": tried}


# --------------------------------------------------------------------------- #
def run_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return 0
    from workload import get
    from workload.traces import all_traces
    w = get(args.workload)
    if args.L_ctx:
        w = w.scaled(L_ctx=args.L_ctx)
    w = w.scaled(steps=max(w.steps, args.warmup + args.steps))
    traces = all_traces(w)
    # the same warm-up and timed steps as the GPU arm, the oracle as it stands
    res = cpu_oracle_rate(w, token_traces(w, traces), warmup=args.warmup, steps=args.steps)
    steps = res["steps"]
    line = {"impl": "reference", "metric": METRIC, "value": res["value"], "unit": "selections/s",
            "n_gpus": args.gpus, "steps": steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * res["seconds"] / res["steps"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
            "data": "synthetic", "config": workload_config(w, args, args.gpus),
            "cpu_baseline": {"kind": "oracle", "cores": 1, "sample": res["sample"],
                             "value": res["value"], "unit": "selections/s"},
            "e2e": {"value": res["value"], "unit": "selections/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------- #
def h2d_probe(dev):
    """Pinned cudaMemcpyAsync host->device, 1 GiB x 20, best of 3 rounds (a
    transient dip must not flatter the fractions): GB/s."""
    import torch
    nbytes = 1 << 30
    hbuf = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    dbuf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    for _ in range(3):
        dbuf.copy_(hbuf, non_blocking=True)
    best_ms = None
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(20):
            dbuf.copy_(hbuf, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        best_ms = ms if best_ms is None else min(best_ms, ms)
    del hbuf, dbuf
    return 20 * nbytes / (best_ms / 1e3) / 1e9


def measure(o, w, dev, h2d_gbs, dist=None, world=1, headline=False, rank=0, clocks=None):
    """One workload on this GPU: set-up, step graphs, burn-in, the timed pass,
    per-launch windows, the oracle check of the timed run; with `headline`
    also the repeats, the end-to-end pass, the all-hit and admission figures
    and the burn-in over another trace.  Returns the figures as a dict."""
    import numpy as np
    import torch

    from host_offload_serving_gb300 import hisparse as H
    from host_offload_serving_gb300.runtime import HiSparse, WorkloadMemory, DecodeStep, sm_copy
    from host_offload_serving_gb300.replicas import max_over_ranks, job_throughput
    from workload import records as REC
    from workload.traces import all_traces

    K, W = o.steps, o.warmup
    T = W + K
    if T > w.steps:
        w = w.scaled(steps=T)
    t_setup = time.perf_counter()
    mem = WorkloadMemory(w.R, w.L, w.B, w.P, w.rec, mirror=o.mirror,
                         pool_kind=H.HOST_HUGE if o.pool == "huge" else H.HOST_PINNED,
                         group=(1 + w.followers) if o.interleave else 1)
    REC.fill_host_pool(w, mem.geometry)
    if o.mirror:
        mem.fill_mirror()
    hs = HiSparse(w.R, w.L, w.k, w.B, w.P, w.rec, mem.layer_buffers(), anchor_of=w.anchor_of(),
                  ctas_per_request=o.ctas, replay_ctas=o.replay_ctas, lookup=o.lookup)
    if o.l2_persist:
        hs.set_l2_persisting(o.l2_persist << 20)
    info = hs.info()
    hp_frac = mem.pool.hugepage_fraction()

    def thp_splits():
        d = {}
        try:
            for line in open("/proc/vmstat"):
                k_, v = line.split()
                if k_ in ("thp_split_page", "thp_split_pmd"):
                    d[k_] = int(v)
        except OSError:
            pass
        return d
    splits0 = thp_splits()
    anchor_of = w.anchor_of()
    groups = [(a, [l for l in range(w.L) if anchor_of[l] == a]) for a in w.anchors()]
    G = len(groups)
    if o.verify_rows > 1:   # speculative verify rows, resolved as one union list
        from workload.traces import verify_row_traces
        trace_of = lambda ww: verify_row_traces(ww, o.verify_rows)  # noqa: E731
    else:
        trace_of = all_traces
    traces = trace_of(w)
    sel_np = np.stack([traces[a][0] for a, _ in groups], axis=1)       # [T][G][R][k]
    sel = torch.from_numpy(sel_np).to(dev)
    # another trace over the same pool (another selection seed), for a burn-in
    # that does not touch exactly the timed accesses
    sel_alt = None
    if headline and not o.no_burn_in and not o.no_alt_burn_in:
        tr_alt = trace_of(w.scaled(seed=w.seed + 7919))
        sel_alt = torch.from_numpy(np.stack([tr_alt[a][0] for a, _ in groups], axis=1)).to(dev)
    newest = newest_np = wb = new_rows = None
    if w.write_through:
        newest_np = traces[groups[0][0]][1]
        newest = torch.from_numpy(newest_np).to(dev)
        wbn = np.full((w.steps, w.L, w.R), -1, np.int32)
        for t in range(1, w.steps):
            wbn[t] = newest_np[t - 1][None, :]
        wb = torch.from_numpy(wbn).to(dev)
        new_rows = torch.from_numpy(REC.new_token_records(w)).to(dev)
    out = torch.full((G, w.R, w.k), -1, dtype=torch.int32, device=dev)
    seq_dev = None
    if w.admit_preload:   # short requests: admitted preloaded, resolved with their lengths
        seq_dev = torch.from_numpy(np.ascontiguousarray(
            (w.L_ctx + 1 + np.arange(w.steps, dtype=np.int32))[:, None].repeat(w.R, axis=1))).to(dev)
    admit_reqs = torch.arange(w.R, dtype=torch.int32, device=dev)
    admit_pre = torch.full((w.R,), w.L_ctx, dtype=torch.int32, device=dev)

    def admit_all():
        if w.admit_preload:
            hs.admit(-1, admit_reqs, admit_pre)

    admit_all()
    runner = DecodeStep(hs, mem, groups,
                        flags=(H.FROM_MIRROR if o.mirror else 0) |
                        (H.UNION if o.verify_rows > 1 else 0) |
                        (H.SKIP_IO if o.skip_io else 0),
                        fused=not o.unfused, sel_block_tokens=w.sel_block_tokens,
                        group_replay=o.replay == "group", inline_shared=o.replay == "inline")
    miss_hist = torch.zeros((T, G, w.R), dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)     # > 129 MB L2
    setup_s = time.perf_counter() - t_setup

    res_all = res_tok = None
    if o.resident:
        from workload.resident import resident_tables
        full, window, tok = (int(x) for x in o.resident.split(","))
        res_all = torch.from_numpy(resident_tables(w, tok, full=full, window=window)).to(dev)
        res_tok = tok

    def issue(t, sel_src=None):
        s = sel if sel_src is None else sel_src
        if res_all is not None:          # step t's resident block table, by pointer
            runner.resident = (res_all[t], res_tok)
        runner.issue(s[t], out, newest=newest[t] if newest is not None else None,
                     wb_pos=wb[t] if (wb is not None and t > 0) else None,
                     new_rows=new_rows[t] if new_rows is not None else None,
                     seq_lens=seq_dev[t] if seq_dev is not None else None)

    # Every step is captured once as a CUDA graph -- the form the pages deploy
    # RESOLVE in (gentlecold.top deep dive §3.5: captured in the decode CUDA
    # graph) -- so the timed region measures GPU work, not Python launch
    # overhead.
    def timing_event():
        try:
            return torch.cuda.Event(enable_timing=True, external=True), True
        except TypeError:
            return torch.cuda.Event(enable_timing=True), False

    cap = torch.cuda.Stream()

    def capture(t, instrument, sel_src=None):
        """Graph of step t; with `instrument`, timing events around every
        RESOLVE, write-back and replay launch and a copy of the miss counts."""
        evs, wev, rpev = [], [], []
        names = ("resolve", "resolve_step", "resolve_resident", "resolve_ex", "writeback",
                 "prefetch_plan")
        orig = {n: getattr(hs, n) for n in names}

        def timed(fn, acc):
            def call(*a, **kw):
                st = kw.get("stream")
                e0, e1 = timing_event()[0], timing_event()[0]
                e0.record(st)
                fn(*a, **kw)
                e1.record(st)
                acc.append((e0, e1))
            return call

        if instrument:
            for n in names[:4]:
                setattr(hs, n, timed(orig[n], evs))
            hs.writeback = timed(orig["writeback"], wev)
            hs.prefetch_plan = timed(orig["prefetch_plan"], rpev)
        g = torch.cuda.CUDAGraph()
        try:
            with torch.cuda.stream(cap):
                with torch.cuda.graph(g, stream=cap):
                    issue(t, sel_src)
                    if instrument:
                        for gi, (a, _) in enumerate(groups):
                            hs.copy_miss_counts(a, miss_hist[t, gi],
                                                stream=torch.cuda.current_stream())
        finally:
            for n in names:
                setattr(hs, n, orig[n])
        return g, evs, wev, rpev

    def capture_pass(events):
        """One graph holding the K timed steps, each after the L2 flush; with
        `events`, a pair of CUDA events inside the graph around each step.  The
        pass is one graph launch, so no timed step carries a graph launch of
        its own (as in a serving step, whose graph holds every layer)."""
        evs = [(timing_event()[0], timing_event()[0]) for _ in range(K)] if events else None
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                s = torch.cuda.current_stream()
                for i in range(K):
                    flush.fill_(i & 0xFF)
                    if events:
                        evs[i][0].record(s)
                    issue(W + i)
                    if events:
                        evs[i][1].record(s)
        return g, evs

    def capture_flush_only():
        """The pass graph without the steps: K L2 flushes."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                for i in range(K):
                    flush.fill_(i & 0xFF)
        return g

    ext_ok = timing_event()[1]
    plain = [capture(t, False)[0] for t in range(T)]
    plain_alt = [capture(t, False, sel_alt)[0] for t in range(T)] if sel_alt is not None else None
    instr = [capture(t, ext_ok) for t in range(T)] if ext_ok else None
    passg = capture_pass(True) if ext_ok else None
    pass_net = capture_pass(False)
    flush_g = capture_flush_only()
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream()

    def wake():
        """About 2 ms of HBM writes before the warm-up, so that the timed steps
        do not start on a GPU that sat idle while the host prepared them (a
        serving GPU is busy step after step)."""
        for i in range(40):
            flush.fill_(i & 0xFF)

    def from_admission(warm=True):
        hs.reset()
        mem.hot.zero_()
        admit_all()
        torch.cuda.synchronize()
        if warm:
            wake()
            for t in range(W):
                plain[t].replay()
            torch.cuda.synchronize()

    def burn(graphs):
        """Untimed passes over every step, each from the admission state.  The
        GPU's first accesses to host pages of a new pool pay one-time
        address-translation work (tens of us to ms per launch, measured to last
        about two passes over a trace); a serving system pays that once at
        start-up, so it stays out of the timed steps."""
        for _ in range(0 if o.no_burn_in else o.burn_in):
            for t in range(T):
                graphs[t].replay()
            torch.cuda.synchronize()
            from_admission(warm=False)

    def per_step_graphs():
        """The K timed steps as K graph launches, events outside the graphs
        (each step pays its own graph launch); returns per-step ms."""
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)]
        for i in range(K):
            flush.fill_(i & 0xFF)     # also keeps the GPU busy while the host enqueues
            ev[i][0].record(cur)
            plain[W + i].replay()
            ev[i][1].record(cur)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in ev]

    def timed_pass():
        """Pass 1: per-step ms (events inside the pass graph around each step)."""
        if passg is not None:
            passg[0].replay()
            torch.cuda.synchronize()
            return [a.elapsed_time(b) for a, b in passg[1]]
        return per_step_graphs()     # no timing events inside graphs in this torch

    def net_pass():
        """The K steps without any event between them, minus the same graph
        with the flushes alone: ms per step of the steps' own GPU time."""
        res = []
        for _ in range(3):
            from_admission()
            e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            e[0].record(cur)
            pass_net[0].replay()
            e[1].record(cur)
            e[2].record(cur)
            flush_g.replay()
            e[3].record(cur)
            torch.cuda.synchronize()
            res.append((e[0].elapsed_time(e[1]) - e[2].elapsed_time(e[3])) / K)
        return sorted(res)[1], res

    # ---- burn-in over another trace, then the timed steps (headline only):
    #      the timed accesses are then not the ones the burn-in warmed ----
    alt = None
    if plain_alt is not None:
        burn(plain_alt)
        from_admission()
        alt_ms = timed_pass()
        alt = {"ms_per_step": round(sum(alt_ms) / K, 4),
               "selections_per_s": round(G * w.R * w.k * K / (sum(alt_ms) / 1e3), 1),
               "burn_in": f"{o.burn_in} passes over a trace of another selection seed on "
                          "the same pool, then the W warm-up and K timed steps of the "
                          "timed trace"}
        from_admission(warm=False)

    # ---- burn-in over the timed trace, then pass 1 (the headline): W warm-up
    #      steps, then exactly K timed steps, the L2 flushed before each, all
    #      K in one graph launch with an event pair inside the graph around
    #      every step ----
    if clocks is not None:   # sampling from before the burn-in until after the timed pass
        clocks.__enter__()
        t_wait = time.time()
        while not clocks.samples and time.time() - t_wait < 5:
            time.sleep(0.05)
    burn(plain)
    splits_burn = {k_: v - splits0.get(k_, 0) for k_, v in thp_splits().items()}
    splits0 = thp_splits()
    from_admission()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    step_ms = timed_pass()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    if clocks is not None:
        time.sleep(0.25)           # one more clock sample after the timed region
        clocks.__exit__()
    flags, _ = hs.status()

    replay_launches = sum((-(-len(f) // 8) if o.replay == "group" else
                           0 if o.replay == "inline" else len(f)) for _, f in groups if f)
    launches = K * (G + replay_launches + (1 if (wb is not None and o.unfused) else 0))

    rep_ms = sg_ms = None
    # the whole trace more times from the admission state, timed like pass 1
    rep_ms = []
    for _ in range(5 if headline else 3):
        from_admission()
        rep_ms.append(sum(timed_pass()) / K)
    if headline:
        # one graph launch per step (the difference is the graph launch)
        from_admission()
        sg_ms = per_step_graphs()
    net_ms, net_all = net_pass()

    # ---- pass 2 (per-kernel durations): the same steps from the admission
    #      state, with events inside the graphs around every launch ----
    from_admission(warm=False)
    res_ms = wb_ms = rp_ms = cold_ms = None
    if instr is not None:
        for t in range(T):
            flush.fill_(t & 0xFF)
            instr[t][0].replay()
            torch.cuda.synchronize()
        res_ms = [[a.elapsed_time(b) for a, b in instr[W + i][1]] for i in range(K)]
        cold_ms = [a.elapsed_time(b) for a, b in instr[0][1]]
        wb_ms = [a.elapsed_time(b) for i in range(K) for a, b in instr[W + i][2]]
        rp_ms = [a.elapsed_time(b) for i in range(K) for a, b in instr[W + i][3]]
    else:   # no in-graph timing events in this torch: count misses eagerly
        for t in range(T):
            plain[t].replay()
            for gi, (a, _) in enumerate(groups):
                hs.copy_miss_counts(a, miss_hist[t, gi], stream=cur)
        torch.cuda.synchronize()
    flags |= hs.status()[0]
    miss = miss_hist[W:].cpu().numpy().astype(np.int64)       # [K][G][R]
    # ---- the timed steps' final state against the oracle (pass 2 ran the same
    #      steps from the admission state, so the state is the timed run's).
    #      Checked after all GPU timing: the host work of the check can make
    #      the GPU drop its translations of the host pool, which slows the next
    #      pass. ----
    verify = None
    if o.verify and not o.resident and w.sel_block_tokens == 1 and o.verify_rows == 1:
        verify = verify_against_oracle(w, hs, mem, groups, traces, T,
                                       check_bytes=not o.skip_io)

    total_ms = sum(step_ms)
    sel_per_step = G * w.R * w.k
    total_ms_max = max_over_ranks(total_ms, dist, dev)
    value = job_throughput(sel_per_step * K, total_ms_max / 1e3, world)

    if res_ms is not None:
        res_flat = [x for r in res_ms for x in r]
    else:
        res_flat = [x / G for x in step_ms]
    resolve_avg_ms = sum(res_flat) / len(res_flat)
    srt = sorted(res_flat)
    pct = lambda q: srt[min(len(srt) - 1, int(q * (len(srt) - 1) + 0.5))] * 1e3  # noqa: E731
    # When a step holds nothing but the RESOLVE launches (write-through fused,
    # no replay launches), a launch's duration is the step time over the
    # launches per step: from pass 1 (events around each step) and from the
    # event-free pass (the steps' own GPU time).
    inline = o.replay == "inline"
    only_resolve = (all(not f for _, f in groups) or (inline and wb is None)) and \
        not (o.unfused and wb is not None)
    if only_resolve:
        launch_ms = (total_ms / K) / G
        launch_net_ms = net_ms / G
        timing_note = ("launch = step time / RESOLVE launches per step (the step holds only "
                       "RESOLVE launches). avg_launch_us: the event-free pass (the K steps in "
                       "one graph with no event between them, minus the same graph with the "
                       "L2 flushes alone; median of 3). avg_launch_us_step_events: pass 1, "
                       "CUDA events inside the pass graph around each step (each step then "
                       "also carries its two events' idle time). Percentiles: per-launch event "
                       "windows in a second pass over the same steps")
    else:
        launch_ms = resolve_avg_ms
        launch_net_ms = None
        timing_note = ("launch = per-launch event windows in a second pass over the same steps "
                       "(the step also holds replay or write-back launches)")
    miss_bytes = int(miss.sum()) * w.rec
    if inline:   # a RESOLVE launch also moves every miss's rows of its shared-index layers
        miss_bytes = sum(int(miss[:, gi].sum()) * (1 + len(f))
                         for gi, (_, f) in enumerate(groups)) * w.rec
    n_launch = K * G
    fetch_gbs = miss_bytes / (launch_ms * n_launch / 1e3) / 1e9
    fetch_net_gbs = (miss_bytes / (launch_net_ms * n_launch / 1e3) / 1e9
                     if launch_net_ms else None)
    miss_rate = float(miss.sum()) / (K * G * w.R * w.k)

    cold = None
    if cold_ms:
        cb = int(miss_hist[0].sum().item()) * w.rec
        if inline:
            cb = sum(int(miss_hist[0, gi].sum().item()) * (1 + len(f))
                     for gi, (_, f) in enumerate(groups)) * w.rec
        c_s = sum(cold_ms) / 1e3
        cold = {"us_per_launch": round(1e3 * sum(cold_ms) / len(cold_ms), 2),
                "bytes_per_launch": cb // G, "fetch_gbs": round(cb / c_s / 1e9, 2),
                "frac_of_link": round(cb / c_s / 1e9 / h2d_gbs, 4),
                "timing": "step 0 of pass 2 (admission state), events around each RESOLVE"}
    replay = None
    if rp_ms:
        nf = sum(len(f) for _, f in groups)
        rp_bytes = sum(int(miss[:, gi].sum()) * len(f) for gi, (_, f) in enumerate(groups)) * w.rec
        replay = {"kernel": "replay_kernel", "launches": len(rp_ms),
                  "us_avg": round(1e3 * sum(rp_ms) / len(rp_ms), 2),
                  "fetch_gbs": round(rp_bytes / (sum(rp_ms) / 1e3) / 1e9, 2),
                  "frac_of_link": round(rp_bytes / (sum(rp_ms) / 1e3) / 1e9 / h2d_gbs, 4),
                  "followers_per_step": nf,
                  "layers_per_launch": round(nf * K / len(rp_ms), 2),
                  "order": "each CTA batch of plan records read in source-address order"}

    # algorithmic HBM bytes of one RESOLVE launch (the metadata side): per unit
    # 4k selections + 4k slot vector + 4B slot map + 2B + 2B LRU order in and
    # out + 12 per miss (slot map and two page-table writes) + the missed
    # records written into the hot buffer; this design also gathers one 4-byte
    # page-table entry per selection
    Mbar = int(miss.sum()) / n_launch
    hbm_alg = (w.R * (4 * w.k + 4 * w.k + 4 * w.B + 2 * w.B + 2 * w.B) + Mbar * (12 + w.rec)
               + (2 * w.R * w.rec if w.write_through else 0))
    hbm_peak = measured_peaks()[0]["hbm_gbs"]
    hbm_gbs = hbm_alg / ((launch_net_ms or launch_ms) / 1e3) / 1e9
    fig = {
        "workload": w.name, "steps": K, "warmup": W,
        "selections_per_s": round(value, 1), "ms_per_step": round(total_ms_max / K, 4),
        "ms_per_step_net": round(net_ms, 4),
        "ms_per_step_repeats": [round(x, 4) for x in rep_ms],
        "ms_per_step_net_runs": [round(x, 4) for x in net_all],
        "us_per_layer_step": round(launch_ms * 1e3, 2),
        "us_per_layer_step_net": round(launch_net_ms * 1e3, 2) if launch_net_ms else None,
        "launch_us_p50_p90_p99_max": [round(pct(0.5), 2), round(pct(0.9), 2),
                                      round(pct(0.99), 2), round(srt[-1] * 1e3, 2)],
        "avg_launch_us_event_window": round(resolve_avg_ms * 1e3, 2),
        "miss_rate": round(miss_rate, 4),
        "miss_bytes_per_launch": miss_bytes / n_launch,
        "fetch_gbs": round(fetch_gbs, 2), "fetch_frac_of_link": round(fetch_gbs / h2d_gbs, 4),
        "fetch_gbs_net": round(fetch_net_gbs, 2) if fetch_net_gbs else None,
        "fetch_frac_of_link_net": round(fetch_net_gbs / h2d_gbs, 4) if fetch_net_gbs else None,
        "hbm_algorithmic_bytes_per_launch": round(hbm_alg),
        "hbm_gbs": round(hbm_gbs, 2), "hbm_frac": round(hbm_gbs / hbm_peak, 5),
        "cold_step0": cold, "replay": replay, "verify": verify, "status_flags": flags,
        "setup_s": round(setup_s, 1), "host_pool_gb": round(w.host_bytes() / 1e9, 1),
        "timing": timing_note,
        "_launch_ms": launch_ms, "_launch_net_ms": launch_net_ms, "_miss_bytes": miss_bytes,
        "_launches": launches, "_total_ms_max": total_ms_max,
    }
    if headline:
        fig.update({
            "info": info, "wb_ms": wb_ms, "burn_in_other_trace": alt,
            "repeats": {"ms_per_step": [round(x, 4) for x in rep_ms],
                        "median_ms_per_step": round(sorted(rep_ms)[len(rep_ms) // 2], 4),
                        "timing": "the whole trace 5 more times from the admission state, "
                                  "timed like pass 1 (sub-workloads: 3 times)"},
            "step_graphs": {"ms_per_step": round(sum(sg_ms) / len(sg_ms), 4),
                            "selections_per_s": round(sel_per_step * len(sg_ms) /
                                                      (sum(sg_ms) / 1e3), 1),
                            "timing": "the same steps from the admission state, one graph "
                                      "launch per step, events outside the graphs: adds each "
                                      "step's graph launch to its time"},
            "timing_pass": ("pass graph: the K timed steps in one graph launch, the L2 flush "
                            "before each step, CUDA events recorded inside the graph around "
                            "each step" if passg is not None else
                            "one graph launch per step, events outside"),
            "host_pool_hugepage_fraction": round(hp_frac, 3),
            "host_thp_splits_during_burn_in": splits_burn,
        })
        fig["all_hit_no_io"] = all_hit(o, w, hs, groups, sel, newest, out, flush, cap, cur, G)
        fig["e2e"] = None if o.no_e2e else end_to_end(
            o, w, hs, mem, runner, sel_np, newest_np, wb, out, flush, cap, cur, T, world,
            sm_copy, res_all, res_tok, seq_dev, admit_all)
        fig["admission"] = admission(w, hs, flush, cur, dev, h2d_gbs)
        flags |= hs.status()[0]
        fig["status_flags"] = flags
        fig["host_pool_hugepage_fraction_end"] = round(mem.pool.hugepage_fraction(), 3)
        s1 = thp_splits()
        fig["host_thp_splits_during_run"] = {k_: s1[k_] - splits0.get(k_, 0) for k_ in s1}

    # ---- the oracle on the host cores, on a bounded sample ----
    if rank == 0 and not o.no_cpu and not o.resident:
        views = {l: mem.host_view(l) for l in range(w.L)}
        ttr = token_traces(w, traces)
        uni = o.verify_rows > 1
        cpu = cpu_oracle_rate(w, ttr, host_views=views, budget_s=20.0 if headline else 5.0,
                              union=uni)
        cpu.pop("seconds", None)
        cpu.pop("steps", None)
        fig["cpu_baseline"] = cpu
        if headline:
            cpu_mt = cpu_oracle_rate_threads(w, ttr, views, os.cpu_count() or 1, union=uni)
            cpu_mt.pop("seconds", None)
            fig["cpu_baseline_threads"] = cpu_mt
    hs.close()
    mem.close()
    del plain, plain_alt, instr, passg, pass_net, flush_g
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return fig


def all_hit(o, w, hs, groups, sel, newest, out, flush, cap, cur, G):
    """All-hit / no-IO: the last step's selections again, with SKIP_IO.  Every
    selection is now resident, so this is the metadata path alone (lookup,
    scans, publish) against HBM."""
    import numpy as np
    import torch
    from host_offload_serving_gb300 import hisparse as H
    if o.no_allhit:
        return None
    t_last = o.warmup + o.steps - 1
    gh = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(gh, stream=cap):
            for gi, (a, _) in enumerate(groups):
                hs.resolve_ex(a, sel[t_last, gi], out[gi], None,
                              newest[t_last] if newest is not None else None,
                              sel_block_tokens=w.sel_block_tokens,
                              flags=H.SKIP_IO | (H.UNION if o.verify_rows > 1 else 0),
                              stream=torch.cuda.current_stream())
    torch.cuda.synchronize()
    hit_ms = []
    for i in range(10):
        flush.fill_(i)
        h0, h1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        h0.record(cur)
        gh.replay()
        h1.record(cur)
        torch.cuda.synchronize()
        hit_ms.append(h0.elapsed_time(h1) / G)
    mc = np.stack([hs.export_state(a)[3] for a, _ in groups])
    hit_avg = sum(hit_ms) / len(hit_ms)
    alg = w.R * (4 * w.k + 4 * w.B + 2 * w.B + 2 * w.B + 4 * w.k)   # bytes per launch
    peaks, peak_src = measured_peaks()
    gbs = alg / (hit_avg / 1e3) / 1e9
    return {"us_per_layer_step": round(hit_avg * 1e3, 2), "misses": int(mc.sum()),
            "selections_per_s": round(w.R * w.k / (hit_avg / 1e3), 1),
            "algorithmic_bytes_per_launch": alg, "hbm_gbs": round(gbs, 3),
            "hbm_peak_gbs": peaks.get("hbm_gbs"),
            "hbm_frac": round(gbs / peaks.get("hbm_gbs"), 5),
            "hbm_peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)",
            "timing": "graph of one SKIP_IO resolve per anchor, time / anchors"}


def end_to_end(o, w, hs, mem, runner, sel_np, newest_np, wb, out, flush, cap, cur, T, world,
               sm_copy, res_all, res_tok, seq_dev, admit_all):
    """End to end through the C ABI with host buffers: every step copies its
    selections (and write-back positions, new-token KV) from pinned host
    memory and reads the slot vectors back, inside the timed region.  Steps
    are captured as graphs, as a serving loop would."""
    import numpy as np
    import torch
    from workload import records as REC
    G = sel_np.shape[1]
    # A step's inputs (selections; with write-through also the newest
    # positions, the write-back positions and the new tokens' KV) travel packed
    # in one pinned buffer: one host-to-device copy per step, then the RESOLVE
    # launches, then one device-to-host copy of the slot vectors.
    parts = [("sel", tuple(sel_np.shape[1:]), 4)]
    if w.write_through:
        parts += [("newest", (w.R,), 4), ("wb", (w.L, w.R), 4), ("new", (w.L, w.R, w.rec), 1)]
    offs, off = {}, 0
    for name, shape, isz in parts:
        offs[name] = off
        off += -(-int(np.prod(shape)) * isz // 16) * 16
    h_pack = torch.zeros((T, off), dtype=torch.uint8).pin_memory()
    d_pack = torch.empty(off, dtype=torch.uint8, device=out.device)

    def view(buf, name):
        shape, isz = next((sh, z) for n, sh, z in parts if n == name)
        nb = int(np.prod(shape)) * isz
        return buf[offs[name]:offs[name] + nb].view(torch.int32 if isz == 4 else torch.uint8).view(shape)

    h_new = REC.new_token_records(w) if w.write_through else None
    wb_np = wb.cpu().numpy() if w.write_through else None
    for t in range(T):
        view(h_pack[t], "sel").copy_(torch.from_numpy(sel_np[t]))
        if w.write_through:
            view(h_pack[t], "newest").copy_(torch.from_numpy(newest_np[t]))
            view(h_pack[t], "wb").copy_(torch.from_numpy(wb_np[t]))
            view(h_pack[t], "new").copy_(torch.from_numpy(h_new[t]))
    h_out = torch.empty((T, G, w.R, w.k), dtype=torch.int32).pin_memory()
    wt = w.write_through
    e_graphs = []
    for t in range(T):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                if o.e2e_copy == "sm":
                    sm_copy(d_pack, h_pack[t])
                else:
                    d_pack.copy_(h_pack[t], non_blocking=True)
                if res_all is not None:
                    runner.resident = (res_all[t], res_tok)
                runner.issue(view(d_pack, "sel"), out,
                             newest=view(d_pack, "newest") if wt else None,
                             wb_pos=view(d_pack, "wb") if (wt and t > 0) else None,
                             new_rows=view(d_pack, "new") if wt else None,
                             seq_lens=seq_dev[t] if seq_dev is not None else None)
                if o.e2e_copy == "sm":
                    sm_copy(h_out[t], out)
                else:
                    h_out[t].copy_(out, non_blocking=True)
        e_graphs.append(g)

    def reset():
        hs.reset()
        mem.hot.zero_()
        admit_all()
        torch.cuda.synchronize()
    for _ in range(0 if o.no_burn_in else o.burn_in):   # as for pass 1
        reset()
        for t in range(T):
            e_graphs[t].replay()
        torch.cuda.synchronize()
    reset()
    e2e_ms = []
    for t in range(T):
        if t >= o.warmup:
            flush.fill_(t & 0xFF)
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record(cur)
        e_graphs[t].replay()
        if t >= o.warmup:
            s1.record(cur)
            torch.cuda.synchronize()
            e2e_ms.append(s0.elapsed_time(s1))
    torch.cuda.synchronize()
    sel_per_step = G * w.R * w.k
    return {"value": round(sel_per_step * len(e2e_ms) * world / (sum(e2e_ms) / 1e3), 1),
            "unit": "selections/s", "h2d_bytes_per_step": off,
            "d2h_bytes_per_step": h_out[0].numel() * 4,
            "mode": "per-step CUDA graph built through the C ABI; the step's inputs packed in "
                    "one pinned buffer copied up, and its slot vectors copied back, inside the "
                    "timed region, " + ("by SM threads (hisparse_copy)" if o.e2e_copy == "sm"
                                        else "by the copy engines (cudaMemcpyAsync)")}


def admission(w, hs, flush, cur, dev, h2d_gbs):
    """Every request of every layer reset with its first min(B, P) positions
    preloaded (the short-request path of direct admission), and reset alone
    (the long-request path)."""
    import torch
    reqs_d = torch.arange(w.R, dtype=torch.int32, device=dev)
    npre = min(w.B, w.P)
    pre_d = torch.full((w.R,), npre, dtype=torch.int32, device=dev)
    ms_pre, ms_rst = [], []
    for i in range(5):
        for pre, acc in ((pre_d, ms_pre), (None, ms_rst)):
            flush.fill_(i)
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(cur)
            hs.admit(-1, reqs_d, pre, stream=cur)
            a1.record(cur)
            torch.cuda.synchronize()
            acc.append(a0.elapsed_time(a1))
    ab = w.R * w.L * npre * w.rec
    t_pre = sorted(ms_pre)[len(ms_pre) // 2]
    return {"preload_positions": npre, "bytes": ab,
            "us_preload_all": round(t_pre * 1e3, 1),
            "preload_gbs": round(ab / (t_pre / 1e3) / 1e9, 2),
            "preload_frac_of_link": round(ab / (t_pre / 1e3) / 1e9 / h2d_gbs, 4),
            "us_reset_all": round(sorted(ms_rst)[len(ms_rst) // 2] * 1e3, 1),
            "timing": "hisparse_admit of every request on every layer, median of 5, "
                      "L2 flushed before each"}


def sub_workload(args, name):
    """(workload, options) of one entry of the line's `workloads` object, or
    (None, reason) when it cannot run here."""
    from workload import get, sweep_workload
    base = dict(no_e2e=True, no_allhit=True, resident="", verify_rows=1, unfused=False,
                mirror=False, L_ctx=0)
    if name == "tiny":
        w = get("tiny")
        return w, opts_for(args, replay="group", interleave=False, **base)
    if name == "quest":
        return get("quest"), opts_for(args, replay="group", interleave=False, **base)
    if name == "short":
        return get("short"), opts_for(args, replay="group", interleave=False, **base)
    if name in ("shared_inline", "shared_anchor", "shared_inline_huge"):
        kw = dict(base)
        if name == "shared_inline_huge":   # the same on a huge-page-backed pool
            kw["pool"] = "huge"
        return get("shared"), opts_for(args, replay="group" if name == "shared_anchor"
                                       else "inline", interleave=True, **kw)
    if name in ("sweep", "sweep_huge", "sweep_allhit"):
        B, f = SWEEP_POINT
        L, why = pick_sweep_context(B, f)
        if L is None:
            return None, {"reason": "no capacity-sweep context leaves the host-memory margin",
                          **why}
        w = sweep_workload(B, f, L_ctx=L, all_hit=name == "sweep_allhit")
        if name == "sweep_allhit":   # the HBM mirror of the pool must fit beside the rest
            import torch
            free = torch.cuda.mem_get_info()[0]
            if free < w.host_bytes() + w.hot_bytes() + (16 << 30):
                return None, {"reason": "the HBM mirror does not fit", "hbm_free_gb":
                              round(free / 1e9, 1), "mirror_gb": round(w.host_bytes() / 1e9, 1)}
        kw = dict(base, mirror=name == "sweep_allhit")
        if name == "sweep_huge":   # the same point on a huge-page-backed pool
            kw["pool"] = "huge"
        o = opts_for(args, replay="group", interleave=False, **kw)
        o._context_choice = why
        return w, o
    raise KeyError(name)


def sub_steps(args, w):
    """(warm-up, timed) steps of a workload entry: the bench's, within the
    workload's own step count."""
    W = min(args.warmup, max(3, w.steps // 4))
    return W, max(1, min(args.steps, w.steps - W))


# --------------------------------------------------------------------------- #
def run_ours(args):
    import torch

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from host_offload_serving_gb300.replicas import replica_seed
    from workload import get

    dev = torch.device("cuda", local)
    h2d_gbs = h2d_probe(dev)
    w = get(args.workload)
    if args.L_ctx:
        w = w.scaled(L_ctx=args.L_ctx)
    if w.write_through:
        w = w.scaled(steps=max(w.steps, args.warmup + args.steps))
    w = w.scaled(seed=replica_seed(w.seed, rank))     # each replica its own requests
    clocks = Clocks(local)
    fig = measure(args, w, dev, h2d_gbs, dist=dist, world=world, headline=True, rank=rank,
                  clocks=clocks)

    # ---- the other workloads, each on its own pool (one GPU only) ----
    subs = {}
    names = [] if (args.no_workloads or world > 1) else \
        [n for n in args.workloads.split(",") if n]
    for name in names:
        wo = sub_workload(args, name)
        if wo[0] is None:
            subs[name] = {"skipped": wo[1]}
            continue
        ws, os_ = wo
        Wd, Kd = sub_steps(args, ws)
        os_.warmup, os_.steps = Wd, Kd
        try:
            f = measure(os_, ws, dev, h2d_gbs, rank=rank)
        except Exception as e:   # recorded on the line, the headline stands
            subs[name] = {"error": f"{type(e).__name__}: {e}"}
            torch.cuda.synchronize()
            torch.cuda.empty_cache()
            continue
        for k_ in [k_ for k_ in f if k_.startswith("_")]:
            f.pop(k_)
        f["config"] = workload_config(ws, os_, world)
        if getattr(os_, "_context_choice", None):
            f["context_choice"] = os_._context_choice
        subs[name] = f

    peaks, peak_src = measured_peaks()
    kernel_src = os.path.join(ROOT, "host_offload_serving_gb300", "csrc", "hisparse.cu")
    kname = "resolve_pt_kernel" if args.lookup == 0 else "resolve_kernel"
    prof = profile_traffic(kernel_src, kname)
    K = args.steps
    G = len(w.anchors())
    launch_ms = fig["_launch_net_ms"] or fig["_launch_ms"]
    ach_link = fig["_miss_bytes"] / (launch_ms * K * G / 1e3) / 1e9
    if args.mirror:   # records move HBM -> HBM: read and write once each
        bound, ach, peak = "hbm", 2 * ach_link, peaks["hbm_gbs"]
    else:
        bound, ach, peak = "host_link", ach_link, h2d_gbs
    roof = {"bound": bound, "achieved": round(ach, 2), "peak": round(peak, 2),
            "unit": "GB/s", "frac": round(ach / peak, 4),
            "target_frac": TARGET_LINK_FRAC if bound == "host_link" else None,
            "meets_target": (ach / peak >= TARGET_LINK_FRAC) if bound == "host_link" else None,
            "frac_step_events": round((2 if args.mirror else 1) * fig["_miss_bytes"] /
                                      (fig["_launch_ms"] * K * G / 1e3) / 1e9 / peak, 4),
            "traffic": prof["dram_bytes_per_launch"] if prof else None,
            "traffic_sysmem": prof["sysmem_bytes_per_launch"] if prof else None,
            "traffic_source": prof["source"] if prof else None,
            "traffic_vs": ("dram__bytes_read + dram__bytes_write of one captured launch, against "
                           "hbm_algorithmic_bytes_per_launch (the metadata side and the hot-row "
                           "writes); the host-link reads are traffic_sysmem, against "
                           "algorithmic_bytes_per_launch"),
            "hbm_algorithmic_bytes_per_launch": fig["hbm_algorithmic_bytes_per_launch"],
            "kernel": kname,
            "peak_source": (f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if args.mirror else
                            "pinned cudaMemcpyAsync H2D, 1 GiB x 20, best of 3 rounds, same run"),
            "algorithmic_bytes_per_launch": fig["miss_bytes_per_launch"],
            "avg_launch_us": round(launch_ms * 1e3, 2),
            "avg_launch_us_step_events": round(fig["_launch_ms"] * 1e3, 2),
            "avg_launch_us_event_window": fig["avg_launch_us_event_window"],
            "timing": fig["timing"],
            "launch_us_p50_p90_p99_max": fig["launch_us_p50_p90_p99_max"],
            "writeback_us_avg": (round(1e3 * sum(fig["wb_ms"]) / len(fig["wb_ms"]), 2)
                                 if fig.get("wb_ms") else None)}
    if rank == 0:
        info = fig["info"]
        cfg = workload_config(w, args, world)
        line = {
            "metric": METRIC, "value": fig["selections_per_s"], "unit": "selections/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": fig["ms_per_step"], "ms_per_step_net": fig["ms_per_step_net"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
            "data": "synthetic", "config": cfg,
            "run": {"ctas_per_request": info["ctas_per_request"],
                    "smem_bytes_per_cta": info["smem_bytes"],
                    "metadata_bytes": info["metadata_bytes"],
                    "host_pool_hugepage_fraction": fig["host_pool_hugepage_fraction"],
                    "host_pool_hugepage_fraction_end": fig["host_pool_hugepage_fraction_end"],
                    "host_thp_splits_during_burn_in": fig["host_thp_splits_during_burn_in"],
                    "host_thp_splits_during_run": fig["host_thp_splits_during_run"],
                    "setup_s": fig["setup_s"]},
            "roofline": roof,
            "miss_fetch_gbs": fig["fetch_gbs"], "miss_fetch_gbs_net": fig["fetch_gbs_net"],
            "h2d_link_gbs": round(h2d_gbs, 2), "miss_rate": fig["miss_rate"],
            "us_per_layer_step": fig["us_per_layer_step"],
            "us_per_layer_step_net": fig["us_per_layer_step_net"],
            "all_hit_no_io": fig["all_hit_no_io"],
            "cold_step0": fig["cold_step0"],
            "burn_in_other_trace": fig["burn_in_other_trace"],
            "repeats": fig["repeats"],
            "step_graphs": fig["step_graphs"],
            "timing": fig["timing_pass"],
            "admission": fig["admission"],
            "replay": fig["replay"],
            "e2e": fig["e2e"],
            "cpu_baseline": fig.get("cpu_baseline"),
            "cpu_baseline_threads": fig.get("cpu_baseline_threads"),
            "gpu_launches": fig["_launches"],
            "clocks": clocks.summary(),
            "status_flags": fig["status_flags"],
            "verify": fig["verify"],
            "workloads": subs if names else None,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def verify_against_oracle(w, hs, mem, groups, traces, steps, check_bytes=True):
    """Replay the same steps on the oracle and compare the final state: slot
    maps, LRU orders, page tables and miss counts of every anchor, and (unless
    the run skipped the copies) the bytes of a sample of occupied hot rows of
    every layer against records generated afresh for their positions."""
    import numpy as np
    from oracle.coracle import OracleLayer
    from workload import records as REC
    res = {}
    rng = np.random.default_rng(1)
    hot = mem.hot
    new_rows = REC.new_token_records(w) if w.write_through else None
    ok_all = True
    for a, fl in groups:
        o = OracleLayer(w.R, w.k, w.B, w.P, w.rec, host=mem.host_view(a), host_split=w.L_ctx,
                        keep_bytes=False)
        o.reset()
        if w.admit_preload:
            for r in range(w.R):
                o.admit(r, w.L_ctx, io=False)
        for t in range(steps):
            nw = traces[a][1][t] if w.write_through else None
            if w.admit_preload:
                prev = traces[a][1][t - 1] if t > 0 else np.full(w.R, -1, np.int32)
                o.resolve_with_seq_lens(traces[a][0][t], nw, prev,
                                        np.full(w.R, w.L_ctx + t + 1, np.int32), io=False)
            else:
                o.resolve(traces[a][0][t], nw)
        sp, lru, pt, mc = hs.export_state(a)
        ok = (np.array_equal(sp, o.slot_pos) and np.array_equal(lru, o.lru)
              and np.array_equal(pt, o.page_table) and np.array_equal(mc, o.miss_count))
        # sampled bytes: hot row s of every layer of the group holds the
        # record of the position in slot s
        nbad = nchk = 0
        picks = []
        for r in range(w.R if check_bytes else 0):
            occ = np.flatnonzero(sp[r] >= 0)
            if len(occ):
                picks += [(r, int(s)) for s in rng.choice(occ, size=min(32, len(occ)),
                                                         replace=False)]
        if picks:
            ri = [r for r, _ in picks]
            si = [s for _, s in picks]
            for l in [a] + list(fl):
                got = hot[l][ri, si].cpu().numpy()              # one gather per layer
                for j, (r, s) in enumerate(picks):
                    p = int(sp[r, s])
                    exp = (REC.records(w, l, r, [p])[0] if p < w.L_ctx
                           else new_rows[p - w.L_ctx, l, r])
                    nchk += 1
                    nbad += int(not np.array_equal(got[j], exp))
        res[str(a)] = {"state": bool(ok), "rows_checked": nchk, "rows_differ": nbad}
        ok_all = ok_all and ok and nbad == 0
    res["ok"] = bool(ok_all)
    return res


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
