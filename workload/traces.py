"""Seeded synthetic selection traces (input generation only).

The pages measure on LongBenchV2 selection traces of real models, which are not
available here; these traces stand in for them with the pages' shapes: k
selections per (request, layer, step), strong step-to-step reuse (87% hits at
B=2k is the figure of gentlecold.top "HiSparse 深度解析" §2.3 and §3.3), an
attention sink, a local window that includes the newest token, and a
heavy-tailed remainder.

Recipe for one (request, layer) unit, step t (``Workload`` holds the knobs):
  1. MAND = sink {0..n_sink-1} U local (the last W_loc positions of the
     current context, newest included).
  2. H = union of the previous W_hist steps' selections.
  3. keep_target = floor(f*k + 0.5);
     kept = min(keep_target - |MAND & S_{t-1}|, k - |MAND|), at least 0,
     drawn uniformly without replacement from H minus MAND.
  4. S_t = MAND U kept, filled up to k by Zipf(s) ranks over the prefill
     context (P(rank r) ~ r^-s, inverse CDF on a float64 table) mapped to
     positions by a fixed seeded permutation per unit; repeats are rejected;
     after 64*k rejections the rest is uniform over unselected positions.
  5. The list is a seeded shuffle of S_t.
Step 0 is MAND + Zipf (or uniform distinct positions for ``step0="uniform"``).
With ``write_through`` the newest position at step t is L_ctx + t.
With ``all_hit`` every step repeats step 0's list.
Each unit draws from ``numpy.random.default_rng([seed, layer, request])``.
"""
import numpy as np


def zipf_cdf(N, s):
    w = np.arange(1, N + 1, dtype=np.float64) ** (-float(s))
    c = np.cumsum(w)
    return c / c[-1]


class _ZipfCache:
    def __init__(self):
        self._c = {}

    def get(self, N, s):
        key = (N, float(s))
        if key not in self._c:
            self._c[key] = zipf_cdf(N, s)
        return self._c[key]


_ZC = _ZipfCache()


def unit_trace(w, layer, req):
    """Selections [steps][k] int32 and newest positions [steps] int32 (-1 if none)."""
    rng = np.random.default_rng([w.seed, layer, req])
    k = w.k
    N = w.L_ctx
    cdf = _ZC.get(N, w.zipf_s)
    perm = rng.permutation(N).astype(np.int64)
    P = w.P
    in_s = np.zeros(P, dtype=bool)
    sel = np.empty((w.steps, k), dtype=np.int32)
    newest = np.full(w.steps, -1, dtype=np.int32)
    hist = []
    keep_target = int(np.floor(w.f * k + 0.5))

    for t in range(w.steps):
        if w.all_hit and t > 0:
            sel[t] = sel[0]
            newest[t] = newest[0]
            continue
        nw = w.L_ctx + t if w.write_through else -1
        newest[t] = nw
        ctx_end = nw + 1 if w.write_through else w.L_ctx
        mand = set(range(min(w.n_sink, ctx_end)))
        mand.update(range(max(0, ctx_end - w.W_loc), ctx_end))
        if len(mand) > k:
            raise ValueError("mandatory set larger than k")

        if t == 0 and w.step0 == "uniform":
            S = [int(x) for x in rng.choice(ctx_end, size=k, replace=False)]
        else:
            S = sorted(mand)
            if t > 0:
                prev = hist[-1]
                H = set().union(*hist[-w.W_hist:])
                kept_n = min(keep_target - len(mand & prev), k - len(mand))
                kept_n = max(0, kept_n)
                cand = np.array(sorted(H - mand), dtype=np.int64)
                if kept_n and len(cand):
                    kept = rng.choice(cand, size=min(kept_n, len(cand)), replace=False)
                    S.extend(int(x) for x in kept)
            S = _fill_zipf(rng, S, k, cdf, perm, in_s, ctx_end)
        S = np.array(S, dtype=np.int64)
        sel[t] = rng.permutation(S).astype(np.int32)
        hist.append(set(int(x) for x in S))
        if len(hist) > max(1, w.W_hist):
            hist.pop(0)
    return sel, newest


def _fill_zipf(rng, S, k, cdf, perm, in_s, ctx_end):
    in_s[np.array(S, dtype=np.int64)] = True
    need = k - len(S)
    rejections = 0
    N = len(perm)
    out = list(S)
    while need > 0 and rejections < 64 * k:
        u = rng.random(4096)
        ranks = np.minimum(np.searchsorted(cdf, u, side="right"), N - 1)
        pos = perm[ranks]
        _, first = np.unique(pos, return_index=True)
        first.sort()
        cand = pos[first]
        new = cand[~in_s[cand]]
        take = new[:need]
        rejections += len(pos) - len(new)
        in_s[take] = True
        out.extend(int(x) for x in take)
        need -= len(take)
    if need > 0:
        free = np.flatnonzero(~in_s[:ctx_end])
        take = rng.choice(free, size=need, replace=False)
        in_s[take] = True
        out.extend(int(x) for x in take)
    in_s[np.array(out, dtype=np.int64)] = False
    return out


def layer_traces(w, layer):
    """Selections [steps][R][k] and newest [steps][R] for one RESOLVE layer."""
    sel = np.empty((w.steps, w.R, w.k), dtype=np.int32)
    newest = np.empty((w.steps, w.R), dtype=np.int32)
    for r in range(w.R):
        s, n = unit_trace(w, layer, r)
        sel[:, r, :] = s
        newest[:, r] = n
    return sel, newest


def all_traces(w):
    """{anchor layer: (sel [steps][R][k], newest [steps][R])}.

    For a block-selecting workload (``sel_block_tokens`` = t > 1) the lists
    hold block ids ([steps][R][k / t]): the same recipe run over the context
    in blocks of t positions, with k, the sink and the local window counted
    in blocks."""
    t = w.sel_block_tokens
    if t > 1 and w.write_through:
        raise ValueError("block-selecting workloads here have no write-through (the newest "
                         "token is one position, not a block)")
    if t > 1:
        wb = w.scaled(L_ctx=w.L_ctx // t, k=w.k // t, B=max(w.B // t, w.k // t),
                      n_sink=max(1, w.n_sink // t), W_loc=max(1, w.W_loc // t),
                      sel_block_tokens=1)
        return {l: layer_traces(wb, l) for l in w.anchors()}
    return {l: layer_traces(w, l) for l in w.anchors()}


def verify_row_traces(w, V):
    """Speculative verify rows: {anchor: (sel [steps][R][k], newest)} where each
    request's list is V rows of k / V selections, the row of draft token d at
    step t being the top-k of step t + d of a trace with k / V selections per
    step (so rows overlap as consecutive decode steps do).  The local window is
    capped at a quarter of a row."""
    import numpy as np
    wr = w.scaled(k=w.k // V, steps=w.steps + V - 1, W_loc=min(w.W_loc, w.k // V // 4))
    out = {}
    for a, (sel, nw) in all_traces(wr).items():
        rows = np.concatenate([sel[d:d + w.steps] for d in range(V)], axis=-1)
        out[a] = (np.ascontiguousarray(rows), None if nw is None else nw[:w.steps])
    return out
