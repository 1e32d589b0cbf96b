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
                         "roofline is then against HBM (rows written back later are not "
                         "mirrored)")
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
    ap.add_argument("--verify", action="store_true",
                    help="after timing, compare the final GPU state with the oracle")
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
            "data": "synthetic", "config": {"workload": w.name, "requests": w.R, "layers": w.L,
                                            "top_k": w.k, "B": w.B, "L_ctx": w.L_ctx,
                                            "record_bytes": w.rec},
            "cpu_baseline": {"kind": "oracle", "cores": 1, "sample": res["sample"],
                             "value": res["value"], "unit": "selections/s"},
            "e2e": {"value": res["value"], "unit": "selections/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------- #
def run_ours(args):
    import numpy as np
    import torch

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    from host_offload_serving_gb300 import hisparse as H
    from host_offload_serving_gb300.runtime import HiSparse, WorkloadMemory, DecodeStep, sm_copy
    from workload import get, records as REC, sweep_workload
    from workload.traces import all_traces

    w = get(args.workload)
    if args.L_ctx:
        w = w.scaled(L_ctx=args.L_ctx)
    if w.write_through:
        w = w.scaled(steps=max(w.steps, args.warmup + args.steps))
    from host_offload_serving_gb300.replicas import replica_seed, max_over_ranks, job_throughput
    w = w.scaled(seed=replica_seed(w.seed, rank))     # each replica its own requests
    T = args.warmup + args.steps
    if not w.write_through and T > w.steps:
        w = w.scaled(steps=T)
    dev = torch.device("cuda", local)

    t_setup = time.perf_counter()
    mem = WorkloadMemory(w.R, w.L, w.B, w.P, w.rec, mirror=args.mirror,
                         pool_kind=H.HOST_HUGE if args.pool == "huge" else H.HOST_PINNED,
                         group=(1 + w.followers) if args.interleave else 1)
    REC.fill_host_pool(w, mem.geometry)
    if args.mirror:
        mem.fill_mirror()
    hs = HiSparse(w.R, w.L, w.k, w.B, w.P, w.rec, mem.layer_buffers(), anchor_of=w.anchor_of(),
                  ctas_per_request=args.ctas, replay_ctas=args.replay_ctas, lookup=args.lookup)
    info = hs.info()
    hp_frac = mem.pool.hugepage_fraction()

    def thp_splits():
        d = {}
        try:
            for line in open("/proc/vmstat"):
                k, v = line.split()
                if k in ("thp_split_page", "thp_split_pmd"):
                    d[k] = int(v)
        except OSError:
            pass
        return d
    splits0 = thp_splits()
    anchor_of = w.anchor_of()
    groups = [(a, [l for l in range(w.L) if anchor_of[l] == a]) for a in w.anchors()]
    G = len(groups)
    if args.verify_rows > 1:   # speculative verify rows, resolved as one union list
        from workload.traces import verify_row_traces
        traces = verify_row_traces(w, args.verify_rows)
    else:
        traces = all_traces(w)
    sel_np = np.stack([traces[a][0] for a, _ in groups], axis=1)       # [T][G][R][k]
    sel = torch.from_numpy(sel_np).to(dev)
    newest = newest_np = None
    wb = None
    new_rows = None
    if w.write_through:
        newest_np = traces[groups[0][0]][1]
        newest = torch.from_numpy(newest_np).to(dev)
        wbn = np.full((w.steps, w.L, w.R), -1, np.int32)
        for t in range(1, w.steps):
            wbn[t] = newest_np[t - 1][None, :]
        wb = torch.from_numpy(wbn).to(dev)
        new_rows = torch.from_numpy(REC.new_token_records(w)).to(dev)
    out = torch.full((G, w.R, w.k), -1, dtype=torch.int32, device=dev)
    runner = DecodeStep(hs, mem, groups,
                        flags=(H.FROM_MIRROR if args.mirror else 0) |
                        (H.UNION if args.verify_rows > 1 else 0),
                        fused=not args.unfused, sel_block_tokens=w.sel_block_tokens,
                        group_replay=args.replay == "group",
                        inline_shared=args.replay == "inline")
    miss_hist = torch.zeros((T, G, w.R), dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)     # > 129 MB L2
    setup_s = time.perf_counter() - t_setup

    res_all = None
    if args.resident:
        from workload.resident import resident_tables
        full, window, tok = (int(x) for x in args.resident.split(","))
        res_all = torch.from_numpy(resident_tables(w, tok, full=full, window=window)).to(dev)
        res_tok = tok

    def issue(t):
        if res_all is not None:          # step t's resident block table, by pointer
            runner.resident = (res_all[t], res_tok)
        runner.issue(sel[t], out, newest=newest[t] if newest is not None else None,
                     wb_pos=wb[t] if (wb is not None and t > 0) else None,
                     new_rows=new_rows[t] if new_rows is not None else None)

    # Every step is captured once as a CUDA graph -- the form the pages deploy
    # RESOLVE in (gentlecold.top deep dive §3.5: captured in the decode CUDA
    # graph) -- so the timed region measures GPU work, not Python launch
    # overhead.  The headline pass replays plain graphs; a second pass over the
    # same steps replays graphs with timing events around every RESOLVE and
    # write-back launch, on the stream each runs on.
    def timing_event():
        try:
            return torch.cuda.Event(enable_timing=True, external=True), True
        except TypeError:
            return torch.cuda.Event(enable_timing=True), False

    cap = torch.cuda.Stream()

    def capture(t, instrument):
        """Graph of step t; with `instrument`, timing events around every
        RESOLVE and write-back launch and a copy of the miss counts."""
        evs, wev, rpev = [], [], []
        orig_resolve, orig_step = hs.resolve, hs.resolve_step
        orig_res, orig_ex = hs.resolve_resident, hs.resolve_ex
        orig_wb, orig_rp = hs.writeback, hs.prefetch_plan

        def timed_resolve(layer, *a, **kw):
            st = kw.get("stream")
            e0, e1 = timing_event()[0], timing_event()[0]
            e0.record(st)
            orig_resolve(layer, *a, **kw)
            e1.record(st)
            evs.append((e0, e1))

        def timed_step(layer, *a, **kw):
            st = kw.get("stream")
            e0, e1 = timing_event()[0], timing_event()[0]
            e0.record(st)
            orig_step(layer, *a, **kw)
            e1.record(st)
            evs.append((e0, e1))

        def timed_res(layer, *a, **kw):
            st = kw.get("stream")
            e0, e1 = timing_event()[0], timing_event()[0]
            e0.record(st)
            orig_res(layer, *a, **kw)
            e1.record(st)
            evs.append((e0, e1))

        def timed_ex(layer, *a, **kw):
            st = kw.get("stream")
            e0, e1 = timing_event()[0], timing_event()[0]
            e0.record(st)
            orig_ex(layer, *a, **kw)
            e1.record(st)
            evs.append((e0, e1))

        def timed_wb(layer, *a, **kw):
            st = kw.get("stream")
            e0, e1 = timing_event()[0], timing_event()[0]
            e0.record(st)
            orig_wb(layer, *a, **kw)
            e1.record(st)
            wev.append((e0, e1))

        def timed_rp(anchor, follower, *a, **kw):
            st = kw.get("stream")
            e0, e1 = timing_event()[0], timing_event()[0]
            e0.record(st)
            orig_rp(anchor, follower, *a, **kw)
            e1.record(st)
            rpev.append((e0, e1))

        if instrument:
            hs.resolve, hs.resolve_step = timed_resolve, timed_step
            hs.resolve_resident, hs.resolve_ex = timed_res, timed_ex
            hs.writeback, hs.prefetch_plan = timed_wb, timed_rp
        g = torch.cuda.CUDAGraph()
        try:
            with torch.cuda.stream(cap):
                with torch.cuda.graph(g, stream=cap):
                    issue(t)
                    if instrument:
                        for gi, (a, _) in enumerate(groups):
                            hs.copy_miss_counts(a, miss_hist[t, gi],
                                                stream=torch.cuda.current_stream())
        finally:
            hs.resolve, hs.resolve_step = orig_resolve, orig_step
            hs.resolve_resident, hs.resolve_ex = orig_res, orig_ex
            hs.writeback, hs.prefetch_plan = orig_wb, orig_rp
        return g, evs, wev, rpev

    def capture_pass():
        """One graph holding the K timed steps, each after the L2 flush and
        between two events recorded inside the graph: the pass is one graph
        launch, so no timed step carries a graph launch of its own (as in a
        serving step, whose graph holds every layer of the model)."""
        evs = [(timing_event()[0], timing_event()[0]) for _ in range(args.steps)]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                s = torch.cuda.current_stream()
                for i in range(args.steps):
                    flush.fill_(i & 0xFF)
                    evs[i][0].record(s)
                    issue(args.warmup + i)
                    evs[i][1].record(s)
        return g, evs

    ext_ok = timing_event()[1]
    plain = [capture(t, False)[0] for t in range(T)]
    instr = [capture(t, ext_ok) for t in range(T)] if ext_ok else None
    passg = capture_pass() if ext_ok else None
    torch.cuda.synchronize()

    clocks = Clocks(local)
    clocks.__enter__()
    t_wait = time.time()
    while not clocks.samples and time.time() - t_wait < 5:
        time.sleep(0.05)

    # ---- burn-in: untimed passes over every step on the fresh host pool, each
    #      from the admission state.  The GPU's first accesses to host pages
    #      of a new pool pay one-time address-translation work (tens of us to
    #      ms per launch, measured to last about two passes over a trace); a
    #      serving system pays that once at start-up, so it stays out of the
    #      timed steps. ----
    for _ in range(0 if args.no_burn_in else args.burn_in):
        for t in range(T):
            plain[t].replay()
        torch.cuda.synchronize()
        hs.reset()
        mem.hot.zero_()
        torch.cuda.synchronize()
    splits_burn = {k: v - splits0.get(k, 0) for k, v in thp_splits().items()}
    splits0 = thp_splits()

    cur = torch.cuda.current_stream()

    def per_step_graphs():
        """The K timed steps as K graph launches, events outside the graphs
        (each step pays its own graph launch); returns per-step ms."""
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        for i in range(args.steps):
            flush.fill_(i & 0xFF)     # also keeps the GPU busy while the host enqueues
            ev[i][0].record(cur)
            plain[args.warmup + i].replay()
            ev[i][1].record(cur)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in ev]

    # ---- pass 1 (the headline): W warm-up steps, then exactly K timed steps,
    #      L2 flushed before each, all K in one graph launch with an event pair
    #      inside the graph around every step ----
    for t in range(args.warmup):
        plain[t].replay()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    replay_launches = sum((-(-len(f) // 8) if args.replay == "group" else
                           0 if args.replay == "inline" else len(f))
                          for _, f in groups if f)
    launches = args.steps * (G + replay_launches +
                             (1 if (wb is not None and args.unfused) else 0))
    if passg is not None:
        passg[0].replay()
        torch.cuda.synchronize()
        step_ms = [a.elapsed_time(b) for a, b in passg[1]]
    else:   # no timing events inside graphs in this torch
        step_ms = per_step_graphs()
    if dist is not None:
        dist.barrier()
    time.sleep(0.25)               # one more clock sample after the timed region
    clocks.__exit__()
    flags, _ = hs.status()

    verify = None
    if args.verify and not args.resident and w.sel_block_tokens == 1 and args.verify_rows == 1:
        verify = verify_against_oracle(w, hs, mem, groups, traces, args.warmup + args.steps)

    # ---- repeats: the whole trace 5 more times from the admission state (the
    #      same warm-up and timed steps), so the spread between repeats of the
    #      headline is on the line ----
    def from_admission():
        hs.reset()
        mem.hot.zero_()
        torch.cuda.synchronize()
        for t in range(args.warmup):
            plain[t].replay()
        torch.cuda.synchronize()

    rep_ms = []
    for rep in range(5):
        from_admission()
        if passg is not None:
            passg[0].replay()
            torch.cuda.synchronize()
            rep_ms.append(sum(a.elapsed_time(b) for a, b in passg[1]) / args.steps)
        else:
            rep_ms.append(sum(per_step_graphs()) / args.steps)
    # the same steps once more as one graph launch per step (the timing the
    # headline used before the pass graph; the difference is the graph launch)
    from_admission()
    sg_ms = per_step_graphs()

    # ---- pass 2 (per-kernel durations for the roofline): the same steps from
    #      the admission state, with events inside the graphs around every
    #      RESOLVE and write-back launch ----
    hs.reset()
    mem.hot.zero_()
    torch.cuda.synchronize()
    res_ms = wb_ms = rp_ms = cold_ms = None
    if instr is not None:
        for t in range(T):
            flush.fill_(t & 0xFF)
            instr[t][0].replay()
            torch.cuda.synchronize()
        res_ms = [[a.elapsed_time(b) for a, b in instr[args.warmup + i][1]] for i in range(args.steps)]
        cold_ms = [a.elapsed_time(b) for a, b in instr[0][1]]
        wb_ms = [a.elapsed_time(b) for i in range(args.steps) for a, b in instr[args.warmup + i][2]]
        rp_ms = [a.elapsed_time(b) for i in range(args.steps) for a, b in instr[args.warmup + i][3]]
    else:   # no in-graph timing events in this torch: count misses eagerly
        for t in range(T):
            plain[t].replay()
            for gi, (a, _) in enumerate(groups):
                hs.copy_miss_counts(a, miss_hist[t, gi], stream=cur)
        torch.cuda.synchronize()
    flags |= hs.status()[0]
    miss = miss_hist[args.warmup:].cpu().numpy().astype(np.int64)       # [K][G][R]

    total_ms = sum(step_ms)
    sel_per_step = G * w.R * w.k
    value_local = sel_per_step * args.steps / (total_ms / 1e3)
    total_ms_max = max_over_ranks(total_ms, dist, dev)
    value = job_throughput(sel_per_step * args.steps, total_ms_max / 1e3, world)

    if res_ms is not None:
        res_flat = [x for r in res_ms for x in r]
        timing_note = ("events inside the step graphs around every RESOLVE launch "
                       "(second pass over the same steps)")
    else:   # this torch cannot put timing events inside a graph
        res_flat = [x / G for x in step_ms]
        timing_note = "step graph time / anchors (includes write-back and row copy)"
    resolve_avg_ms = sum(res_flat) / len(res_flat)
    srt = sorted(res_flat)
    pct = lambda q: srt[min(len(srt) - 1, int(q * (len(srt) - 1) + 0.5))] * 1e3
    # When a step graph holds nothing but the RESOLVE launches (write-through
    # fused, no shared-index layers), the average launch over the timed region
    # is the pass-1 step time over the launches per step: the same CUDA events,
    # without the extra event nodes the per-launch windows put between kernels.
    inline = args.replay == "inline"
    only_resolve = (all(not f for _, f in groups) or (inline and wb is None)) and \
        not (args.unfused and wb is not None)
    if only_resolve:
        launch_ms = (sum(step_ms) / len(step_ms)) / G
        timing_note = ("average RESOLVE launch over the timed region = pass-1 step time (CUDA "
                       "events recorded inside the pass graph right before each step's first and "
                       "after its last launch; the step holds only the RESOLVE launches) / "
                       "launches per step; percentiles from per-launch event windows in a second "
                       "pass over the same steps")
    else:
        launch_ms = resolve_avg_ms
    miss_bytes = int(miss.sum()) * w.rec
    if inline:   # a RESOLVE launch also moves every miss's rows of its shared-index layers
        miss_bytes = sum(int(miss[:, gi].sum()) * (1 + len(f))
                         for gi, (_, f) in enumerate(groups)) * w.rec
    fetch_gbs = miss_bytes / (launch_ms * args.steps * G / 1e3) / 1e9
    miss_rate = float(miss.sum()) / (args.steps * G * w.R * w.k)

    # ---- host-link probe: pinned cudaMemcpyAsync H2D, 1 GiB x 20, best of
    #      3 rounds (a transient dip must not flatter the fraction) ----
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
    h2d_gbs = 20 * nbytes / (best_ms / 1e3) / 1e9
    del hbuf, dbuf

    # ---- all-hit / no-IO: the last step's selections again, with SKIP_IO.
    #      Every selection is now resident, so this is the metadata path alone
    #      (hash staging, marking, scans, publish) against HBM. ----
    allhit = None
    if not args.no_allhit:
        t_last = args.warmup + args.steps - 1
        gh = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(gh, stream=cap):
                for gi, (a, _) in enumerate(groups):
                    hs.resolve_ex(a, sel[t_last, gi], out[gi], None,
                                  newest[t_last] if newest is not None else None,
                                  sel_block_tokens=w.sel_block_tokens,
                                  flags=H.SKIP_IO | (H.UNION if args.verify_rows > 1 else 0),
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
        allhit = {"us_per_layer_step": round(hit_avg * 1e3, 2), "misses": int(mc.sum()),
                  "selections_per_s": round(w.R * w.k / (hit_avg / 1e3), 1),
                  "algorithmic_bytes_per_launch": alg,
                  "hbm_gbs": round(alg / (hit_avg / 1e3) / 1e9, 3),
                  "timing": "graph of one SKIP_IO resolve per anchor, time / anchors"}

    # ---- end to end through the C ABI with host buffers: every step copies
    #      its selections (and write-back positions, new-token KV) from pinned
    #      host memory and reads the slot vectors back, inside the timed
    #      region.  Steps are captured as graphs, as a serving loop would. ----
    e2e = None
    if not args.no_e2e:
        # A step's inputs (selections; with write-through also the newest
        # positions, the write-back positions and the new tokens' KV) travel
        # packed in one pinned buffer: one host-to-device copy per step, then
        # the RESOLVE launches, then one device-to-host copy of the slot vectors.
        parts = [("sel", tuple(sel_np.shape[1:]), 4)]
        if w.write_through:
            parts += [("newest", (w.R,), 4), ("wb", (w.L, w.R), 4), ("new", (w.L, w.R, w.rec), 1)]
        offs, o = {}, 0
        for name, shape, isz in parts:
            offs[name] = o
            o += -(-int(np.prod(shape)) * isz // 16) * 16
        h_pack = torch.zeros((T, o), dtype=torch.uint8).pin_memory()
        d_pack = torch.empty(o, dtype=torch.uint8, device=dev)

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
        bi = o
        bo = h_out[0].numel() * 4
        e_graphs = []
        for t in range(T):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(cap):
                with torch.cuda.graph(g, stream=cap):
                    if args.e2e_copy == "sm":
                        sm_copy(d_pack, h_pack[t])
                    else:
                        d_pack.copy_(h_pack[t], non_blocking=True)
                    if res_all is not None:
                        runner.resident = (res_all[t], res_tok)
                    runner.issue(view(d_pack, "sel"), out,
                                 newest=view(d_pack, "newest") if wt else None,
                                 wb_pos=view(d_pack, "wb") if (wt and t > 0) else None,
                                 new_rows=view(d_pack, "new") if wt else None)
                    if args.e2e_copy == "sm":
                        sm_copy(h_out[t], out)
                    else:
                        h_out[t].copy_(out, non_blocking=True)
            e_graphs.append(g)
        for burn in range(0 if args.no_burn_in else args.burn_in):   # as for pass 1
            hs.reset()
            mem.hot.zero_()
            torch.cuda.synchronize()
            for t in range(T):
                e_graphs[t].replay()
            torch.cuda.synchronize()
        hs.reset()
        mem.hot.zero_()
        torch.cuda.synchronize()
        e2e_ms = []
        for t in range(T):
            if t >= args.warmup:
                flush.fill_(t & 0xFF)
                s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                s0.record(cur)
            e_graphs[t].replay()
            if t >= args.warmup:
                s1.record(cur)
                torch.cuda.synchronize()
                e2e_ms.append(s0.elapsed_time(s1))
        torch.cuda.synchronize()
        e2e = {"value": round(sel_per_step * len(e2e_ms) * world / (sum(e2e_ms) / 1e3), 1),
               "unit": "selections/s", "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
               "mode": "per-step CUDA graph built through the C ABI; the step's inputs packed "
                       "in one pinned buffer copied up, and its slot vectors copied back, inside "
                       "the timed region, " + ("by SM threads (hisparse_copy)"
                                              if args.e2e_copy == "sm" else
                                              "by the copy engines (cudaMemcpyAsync)")}
        flags |= hs.status()[0]

    peaks, peak_src = measured_peaks()
    kernel_src = os.path.join(ROOT, "host_offload_serving_gb300", "csrc", "hisparse.cu")
    kname = "resolve_pt_kernel" if args.lookup == 0 else "resolve_kernel"
    prof = profile_traffic(kernel_src, kname)
    if args.mirror:   # records move HBM -> HBM: read and write once each
        bound, ach, peak = "hbm", 2 * fetch_gbs, peaks["hbm_gbs"]
    else:
        bound, ach, peak = "host_link", fetch_gbs, h2d_gbs
    roof = {"bound": bound, "achieved": round(ach, 2), "peak": round(peak, 2),
            "unit": "GB/s", "frac": round(ach / peak, 4),
            "traffic": prof["dram_bytes_per_launch"] if prof else None,
            "traffic_sysmem": prof["sysmem_bytes_per_launch"] if prof else None,
            "traffic_source": prof["source"] if prof else None,
            "traffic_launch_algorithmic_bytes": prof["algorithmic_bytes"] if prof else None,
            "kernel": kname,
            "peak_source": (f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if args.mirror else
                            "pinned cudaMemcpyAsync H2D, 1 GiB x 20, best of 3 rounds, same run"),
            "algorithmic_bytes_per_launch": miss_bytes / (args.steps * G),
            "avg_launch_us": round(launch_ms * 1e3, 2),
            "avg_launch_us_event_window": round(resolve_avg_ms * 1e3, 2), "timing": timing_note,
            "launch_us_p50_p90_p99_max": [round(pct(0.5), 2), round(pct(0.9), 2),
                                          round(pct(0.99), 2), round(srt[-1] * 1e3, 2)],
            "writeback_us_avg": round(1e3 * sum(wb_ms) / len(wb_ms), 2) if wb_ms else None}
    # ---- admission: every request of every layer reset with its first
    #      min(B, P) positions preloaded (the short-request path of direct
    #      admission), and reset alone (the long-request path) ----
    admission = None
    if not args.no_allhit:
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
        admission = {"preload_positions": npre, "bytes": ab,
                     "us_preload_all": round(t_pre * 1e3, 1),
                     "preload_gbs": round(ab / (t_pre / 1e3) / 1e9, 2),
                     "preload_frac_of_link": round(ab / (t_pre / 1e3) / 1e9 / h2d_gbs, 4),
                     "us_reset_all": round(sorted(ms_rst)[len(ms_rst) // 2] * 1e3, 1),
                     "timing": "hisparse_admit of every request on every layer, median of 5, "
                               "L2 flushed before each"}
        flags |= hs.status()[0]

    # step 0 from the admission state: every selection but the newest misses,
    # so each launch moves R x k records -- the fetch path at full size
    cold = None
    if cold_ms:
        cb = int(miss_hist[0].sum().item()) * w.rec
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
                  "layers_per_launch": round(nf * args.steps / len(rp_ms), 2)}
    if allhit:
        allhit["hbm_peak_gbs"] = peaks.get("hbm_gbs")
        allhit["hbm_frac"] = round(allhit["hbm_gbs"] / peaks.get("hbm_gbs"), 5)
        allhit["hbm_peak_source"] = f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"

    cpu = cpu_mt = None
    if rank == 0 and not args.no_cpu and not args.resident:
        views = {l: mem.host_view(l) for l in range(w.L)}
        ttr = token_traces(w, traces)
        uni = args.verify_rows > 1
        cpu = cpu_oracle_rate(w, ttr, host_views=views, budget_s=20.0, union=uni)
        cpu.pop("seconds", None)
        cpu.pop("steps", None)
        cpu_mt = cpu_oracle_rate_threads(w, ttr, views, os.cpu_count() or 1, union=uni)
        cpu_mt.pop("seconds", None)

    hp_frac_end = mem.pool.hugepage_fraction()
    s1 = thp_splits()
    splits_run = {k: s1[k] - splits0.get(k, 0) for k in s1}
    hs.close()
    mem.close()
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "selections/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total_ms_max / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
            "config": {"workload": w.name, "requests": w.R, "layers": w.L, "anchors": G,
                       "top_k": w.k, "B": w.B, "L_ctx": w.L_ctx, "record_bytes": w.rec,
                       "write_through": w.write_through, "parallelism": f"replicas{world}",
                       "l2": "flushed (256 MB write) before every timed step",
                       "ctas_per_request": info["ctas_per_request"],
                       "lookup": ["page_table", "hash"][info["lookup"]],
                       "write_through_launch": "separate" if args.unfused else "fused into RESOLVE",
                       "host_pool": args.pool,
                       "replay_launch": {"group": "one per anchor for all its shared-index layers",
                                         "layer": "one per shared-index layer",
                                         "inline": "none: shared-index layers filled inside "
                                                   "the anchor's RESOLVE"}[args.replay],
                       "host_layout": ("rows of each shared-index group interleaved"
                                       if args.interleave else "one block of rows per layer"),
                       "fetch_source": "HBM mirror of the host pool" if args.mirror else "host pool",
                       "verify_rows": args.verify_rows,
                       "resident_tier": (dict(zip(("full_requests", "window", "tokens_per_block"),
                                                  (int(x) for x in args.resident.split(","))))
                                         if args.resident else None),
                       "host_pool_hugepage_fraction": round(hp_frac, 3),
                       "host_pool_hugepage_fraction_end": round(hp_frac_end, 3),
                       "host_thp_splits_during_burn_in": splits_burn,
                       "host_thp_splits_during_run": splits_run,
                       "burn_in": None if args.no_burn_in else
                       f"{args.burn_in} untimed passes over all steps, each from the admission state"},
            "roofline": roof,
            "miss_fetch_gbs": round(fetch_gbs, 2), "h2d_link_gbs": round(h2d_gbs, 2),
            "miss_rate": round(miss_rate, 4),
            "us_per_layer_step": round(launch_ms * 1e3, 2),
            "all_hit_no_io": allhit,
            "cold_step0": cold,
            "repeats": {"ms_per_step": [round(x, 4) for x in rep_ms],
                        "median_ms_per_step": round(sorted(rep_ms)[len(rep_ms) // 2], 4),
                        "timing": "the whole trace 5 more times from the admission state, "
                                  "timed like pass 1"},
            "step_graphs": {"ms_per_step": round(sum(sg_ms) / len(sg_ms), 4),
                            "selections_per_s": round(sel_per_step * len(sg_ms) / (sum(sg_ms) / 1e3), 1),
                            "timing": "the same steps from the admission state, one graph launch "
                                      "per step, events outside the graphs: adds each step's "
                                      "graph launch to its time"},
            "timing": ("pass graph: the K timed steps in one graph launch, the L2 flush before "
                       "each step, CUDA events recorded inside the graph around each step"
                       if passg is not None else "one graph launch per step, events outside"),
            "admission": admission,
            "replay": replay,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "cpu_baseline_threads": cpu_mt,
            "gpu_launches": launches,
            "clocks": clocks.summary(),
            "status_flags": flags,
            "setup_s": round(setup_s, 1),
            "verify": verify,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def verify_against_oracle(w, hs, mem, groups, traces, steps):
    """Replay the same steps on the oracle and compare the final state (sampled bytes)."""
    import numpy as np
    from oracle.coracle import OracleLayer
    from workload import records as REC
    anchors = [a for a, _ in groups]
    res = {}
    for a in anchors:
        o = OracleLayer(w.R, w.k, w.B, w.P, w.rec, host=mem.host_view(a), host_split=w.L_ctx,
                        keep_bytes=False)
        o.reset()
        for t in range(steps):
            nw = traces[a][1][t] if w.write_through else None
            o.resolve(traces[a][0][t], nw)
        sp, lru, pt, mc = hs.export_state(a)
        ok = (np.array_equal(sp, o.slot_pos) and np.array_equal(lru, o.lru)
              and np.array_equal(pt, o.page_table) and np.array_equal(mc, o.miss_count))
        res[str(a)] = bool(ok)
    return res


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
