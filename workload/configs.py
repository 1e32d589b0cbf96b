"""The synthetic workloads, named by what they are and sized like the pages'.

Each workload has the shape of one of the deployments described for HiSparse
(gentlecold.top "HiSparse 深度解析" §4.1 evaluation table, §4.3 B range,
§5.7 deployment config; naphjohn.github.io "推理系统基础设施手记（六）" §2.1):
top-k token selection with k=2048 and B=2k (DSA models), page selection with
Quest, shared-index layer groups (IndexShare), and long-context capacity
points.  The selection traces are synthetic stand-ins for the LongBenchV2
traces the pages measure on; see ``traces.py`` for the recipe.
"""
from dataclasses import dataclass, field, replace


@dataclass(frozen=True)
class Workload:
    name: str
    R: int              # requests in the decode batch
    groups: int         # layers that run RESOLVE (anchors / independent layers)
    followers: int      # shared-index layers per anchor that replay its plan
    L_ctx: int          # prefilled positions per (request, layer)
    k: int              # selections per (request, layer, step)
    B: int              # LRU slots per (request, layer); row B holds the newest token
    rec: int            # record bytes (one position's KV for one layer)
    steps: int          # decode steps
    write_through: bool  # one new token per step, written back to the host pool
    f: float            # reuse fraction of the previous selection(s)
    W_hist: int         # steps of history the reused part is drawn from
    n_sink: int         # attention-sink positions always selected
    W_loc: int          # local window (last W_loc positions) always selected
    zipf_s: float       # exponent of the Zipf draw for the rest
    step0: str = "zipf"  # "zipf" (sink + local + Zipf) or "uniform"
    all_hit: bool = False  # every step repeats step 0's selection list
    seed: int = 0
    sel_block_tokens: int = 1  # > 1: the selector picks blocks of this many positions
    admit_preload: bool = False  # requests admitted with their prefill preloaded and
                                 # resolved with their sequence lengths (short requests)

    @property
    def L(self):
        """Total layers: anchors plus their shared-index followers."""
        return self.groups * (1 + self.followers)

    @property
    def P(self):
        """Host rows per (request, layer): prefill plus one per decode step."""
        return self.L_ctx + (self.steps if self.write_through else 0)

    def anchor_of(self):
        """Per layer: -1 if it runs RESOLVE itself, else its anchor layer."""
        out = []
        for g in range(self.groups):
            a = g * (1 + self.followers)
            out.append(-1)
            out.extend([a] * self.followers)
        return out

    def anchors(self):
        return [l for l, a in enumerate(self.anchor_of()) if a < 0]

    def host_bytes(self):
        return self.L * self.R * self.P * self.rec

    def hot_bytes(self):
        return self.L * self.R * (self.B + 1) * self.rec

    def scaled(self, **kw):
        return replace(self, **kw)


WORKLOADS = {
    # 1 request x 1 layer, 4096 positions, k=64, B=128, 64 steps.
    "tiny": Workload("tiny", R=1, groups=1, followers=0, L_ctx=4096, k=64, B=128, rec=1152,
                     steps=64, write_through=False, f=0.85, W_hist=1, n_sink=4, W_loc=16,
                     zipf_s=1.1, step0="uniform", seed=101),
    # DSA-style token selection: 8 requests x 4 layers, 128K context, k=2048, B=4096.
    "dsa": Workload("dsa", R=8, groups=4, followers=0, L_ctx=131072, k=2048, B=4096, rec=1152,
                    steps=32, write_through=True, f=0.87, W_hist=4, n_sink=4, W_loc=128,
                    zipf_s=1.1, seed=202),
    # Quest-style page selection: 16 requests x 8 layers, 12800 pages of 32 KB.
    "quest": Workload("quest", R=16, groups=8, followers=0, L_ctx=12800, k=128, B=256,
                      rec=32768, steps=32, write_through=False, f=0.80, W_hist=1, n_sink=0,
                      W_loc=0, zipf_s=1.0, seed=303),
    # Block selections: 8 requests x 4 layers, 128K context, top-512 blocks of 4
    # positions (2048 positions), B=4096 (an NSA-style selector).
    "blocks": Workload("blocks", R=8, groups=4, followers=0, L_ctx=131072, k=2048, B=4096,
                       rec=1152, steps=32, write_through=False, f=0.87, W_hist=4, n_sink=4,
                       W_loc=128, zipf_s=1.1, seed=606, sel_block_tokens=4),
    # Short requests: 8 requests x 4 layers whose contexts fit the buffer (3K
    # positions prefilled, B=4096): admitted with their tokens preloaded, then
    # grown by one token per step and looked up by position.
    "short": Workload("short", R=8, groups=4, followers=0, L_ctx=3072, k=2048, B=4096,
                      rec=1152, steps=32, write_through=True, f=0.87, W_hist=4, n_sink=4,
                      W_loc=128, zipf_s=1.1, seed=707, admit_preload=True),
    # Shared-index groups: 32 requests x 4 groups of (1 anchor + 3 shared layers).
    "shared": Workload("shared", R=32, groups=4, followers=3, L_ctx=131072, k=2048, B=4096,
                       rec=1152, steps=32, write_through=False, f=0.87, W_hist=4, n_sink=4,
                       W_loc=128, zipf_s=1.1, seed=404),
}


def sweep_workload(B, f, L_ctx=1048576, all_hit=False):
    """Capacity-sweep point: 64 requests x 2 layers, 1M context, k=2048."""
    name = f"sweep_B{B}_f{int(round(f * 100))}" + ("_allhit" if all_hit else "")
    return Workload(name, R=64, groups=2, followers=0, L_ctx=L_ctx, k=2048, B=B, rec=1152,
                    steps=16, write_through=False, f=f, W_hist=4, n_sink=0, W_loc=0,
                    zipf_s=1.1, all_hit=all_hit, seed=505 + B + int(round(f * 100)))


SWEEP_B = (2048, 4096, 8192)
SWEEP_F = (0.95, 0.87, 0.70)


def get(name):
    if name in WORKLOADS:
        return WORKLOADS[name]
    if name.startswith("sweep_B"):
        parts = name.split("_")
        B = int(parts[1][1:])
        f = int(parts[2][1:]) / 100.0
        return sweep_workload(B, f, all_hit=name.endswith("_allhit"))
    raise KeyError(name)
