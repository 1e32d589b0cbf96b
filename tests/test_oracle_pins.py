"""The oracle pinned to the pages and to mathematics (CPU only)."""
import random

import numpy as np
import pytest

from oracle.tiny import Unit, optimal_misses, ERR_DUP, ERR_RANGE
import pins
from pins import CUnit, ALL_PINS

MODELS = {"python": Unit, "c": CUnit}


@pytest.mark.parametrize("model", sorted(MODELS))
@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(model, pin):
    pin(MODELS[model])


def test_error_codes_match_between_models():
    from oracle import coracle
    assert (ERR_RANGE, ERR_DUP) == (coracle.ERR_RANGE, coracle.ERR_DUP) == (1, 2)


# ---------------------------------------------------------------------- #
# The brute-force optimum, pinned on its own                              #
# ---------------------------------------------------------------------- #
def belady_min(refs, frames):
    """Belady's MIN for single-page references: evict the page used furthest ahead."""
    mem, faults = set(), 0
    for t, p in enumerate(refs):
        if p in mem:
            continue
        faults += 1
        if len(mem) == frames:
            def nxt(q):
                for u in range(t + 1, len(refs)):
                    if refs[u] == q:
                        return u
                return len(refs) + 1
            mem.remove(max(sorted(mem), key=nxt))
        mem.add(p)
    return faults


def test_optimal_textbook_example():
    # Silberschatz et al., Operating System Concepts: optimal replacement on this
    # reference string with 3 frames takes 9 page faults.
    refs = [7, 0, 1, 2, 0, 3, 0, 4, 2, 3, 0, 3, 2, 1, 2, 0, 1, 7, 0, 1]
    assert optimal_misses([[p] for p in refs], 3) == 9
    assert belady_min(refs, 3) == 9


def test_optimal_matches_belady_min_for_single_page_steps():
    for seed in range(30):
        rnd = random.Random(seed)
        frames = rnd.randint(1, 4)
        refs = [rnd.randrange(7) for _ in range(rnd.randint(3, 14))]
        assert optimal_misses([[p] for p in refs], frames) == belady_min(refs, frames)


def test_optimal_closed_forms():
    rnd = random.Random(7)
    for _ in range(20):
        B = rnd.randint(2, 4)
        trace = [rnd.sample(range(8), rnd.randint(1, B)) for _ in range(rnd.randint(1, 5))]
        distinct = len(set().union(*map(set, trace)))
        # enough room for everything: only the first touch of each position misses
        assert optimal_misses(trace, 8) == distinct
        # every step needs its own positions, and the first step all misses
        assert optimal_misses(trace, B) >= len(set(trace[0]))


# ---------------------------------------------------------------------- #
# Python model == C model, full state, on random traces                   #
# ---------------------------------------------------------------------- #
@pytest.mark.parametrize("union", [False, True])
@pytest.mark.parametrize("resident", [False, True])
@pytest.mark.parametrize("seed", range(12))
def test_python_equals_c(seed, resident, union):
    from oracle.coracle import OracleLayer
    rnd = random.Random(seed)
    R = rnd.randint(1, 3)
    k = rnd.randint(1, 12)
    B = k + rnd.randint(0, 10)
    P = rnd.randint(k + 1, 60)
    rec = 16
    host = np.random.default_rng(seed).integers(0, 256, size=(R, P, rec), dtype=np.uint8)
    py = [Unit(B, P, k=k, host=lambda p, r=r: bytes(host[r, p])) for r in range(R)]
    c = OracleLayer(R, k, B, P, rec, host=host)
    c.reset()
    for t in range(30):
        sel = np.full((R, k), -1, np.int32)
        newest = np.full(R, -1, np.int32)
        for r in range(R):
            n = rnd.randint(0, k)
            S = rnd.sample(range(P), n)
            if rnd.random() < (0.5 if union else 0.08) and n >= 2:
                S[1] = S[0]                      # duplicate (a shared position in union mode)
            if union and n >= 4 and rnd.random() < 0.5:
                S[3] = S[2]
            if rnd.random() < 0.05 and n >= 1:
                S[0] = rnd.choice([P, P + 5, -3])  # out of range
            sel[r, :n] = S
            rnd.shuffle(sel[r])
            if S and rnd.random() < 0.3:
                newest[r] = rnd.choice(S)
        tok, blocks = rnd.choice([1, 2, 4]), None
        if resident:
            nb = rnd.randint(1, P // tok + 1)
            blocks = np.array([[rnd.randrange(200) if rnd.random() < 0.3 else
                                (-1 if rnd.random() < 0.97 else -4) for _ in range(nb)]
                               for _ in range(R)], np.int32)
        out_c, e_c = c.resolve(sel, newest, res_blocks=blocks, res_tok=tok, union=union)
        e_py = 0
        for r in range(R):
            out, plan, err = py[r].resolve([int(x) for x in sel[r]], int(newest[r]),
                                           res_blocks=None if blocks is None else
                                           [int(x) for x in blocks[r]], res_tok=tok,
                                           union=union)
            e_py |= err
            assert out == list(out_c[r]), (t, r)
            assert err == c.unit_err[r]
            assert py[r].slot_pos == list(c.slot_pos[r])
            assert py[r].lru == list(c.lru[r])
            pt = {int(p): int(c.page_table[r, p]) for p in np.flatnonzero(c.page_table[r] >= 0)}
            assert py[r].page_table == pt
            assert py[r].miss_count == c.miss_count[r]
            assert plan == [(int(c.plan_pos[r, j]), int(c.plan_slot[r, j]))
                            for j in range(c.plan_count[r])]
            for s in range(B):
                if py[r].hot[s] is not None:
                    assert py[r].hot[s] == bytes(c.hot[r, s])
        assert e_py == e_c


# ---------------------------------------------------------------------- #
# Write-through and plan replay (C model)                                 #
# ---------------------------------------------------------------------- #
def test_writeback_then_fetch_returns_written_bytes():
    from oracle.coracle import OracleLayer
    R, k, B, L_ctx, steps, rec = 2, 3, 4, 10, 3, 16
    P = L_ctx + steps
    rng = np.random.default_rng(3)
    host = rng.integers(0, 256, size=(R, P, rec), dtype=np.uint8)
    c = OracleLayer(R, k, B, P, rec, host=host, host_split=L_ctx)
    c.reset()
    assert (c.host_tail == 0xA5).all()                 # unwritten rows are poisoned
    newrec = rng.integers(0, 256, size=(steps, R, rec), dtype=np.uint8)
    for t in range(steps):
        if t > 0:
            c.writeback(np.full(R, L_ctx + t - 1, np.int32))
        c.set_newest_rows(newrec[t])
        # select the previous token (now on the host) and the newest one
        sel = np.full((R, k), -1, np.int32)
        sel[:, 0] = L_ctx + t
        if t > 0:
            sel[:, 1] = L_ctx + t - 1
        out, e = c.resolve(sel, np.full(R, L_ctx + t, np.int32))
        assert e == 0
        assert (out[:, 0] == B).all()
        if t > 0:
            for r in range(R):
                assert bytes(c.hot[r, out[r, 1]]) == bytes(newrec[t - 1, r])


def test_replay_follows_anchor_slots():
    from oracle.coracle import OracleLayer
    R, k, B, P, rec = 3, 5, 7, 40, 16
    rng = np.random.default_rng(11)
    host_a = rng.integers(0, 256, size=(R, P, rec), dtype=np.uint8)
    host_f = rng.integers(0, 256, size=(R, P, rec), dtype=np.uint8)
    a = OracleLayer(R, k, B, P, rec, host=host_a)
    f = OracleLayer(R, k, B, P, rec, host=host_f, metadata=False)
    a.reset()
    for t in range(20):
        sel = np.stack([rng.choice(P, size=k, replace=False) for _ in range(R)]).astype(np.int32)
        a.resolve(sel)
        a.replay_into(f)
        for r in range(R):
            for s in range(B):
                p = a.slot_pos[r, s]
                if p >= 0:
                    assert bytes(f.hot[r, s]) == bytes(host_f[r, p])
                    assert bytes(a.hot[r, s]) == bytes(host_a[r, p])


# ---------------------------------------------------------------------- #
# Planted mistakes: each must fail at least one pin                       #
# ---------------------------------------------------------------------- #
class _Mutant(Unit):
    mutation = None

    def resolve(self, sel, newest=-1, skip_io=False, res_blocks=None, res_tok=1, union=False):
        m = self.mutation
        B, P, k = self.B, self.P, len(sel)
        if union and m == "union_last_reference":
            sel = list(sel)
            order = list(range(k))[::-1]      # classify from the end: last reference wins
        else:
            order = list(range(k))

        def rrow(p):
            if res_blocks is None or p // res_tok >= len(res_blocks):
                return -1
            e = res_blocks[p // res_tok]
            if e < -1 and m != "resident_no_entry_check":
                return None
            if e < 0:
                return -1
            row = e * res_tok + (0 if m == "resident_no_offset" else p % res_tok)
            return row if B + 1 + row < 2**31 else None

        err, seen = 0, set()
        for p in sel:
            if p == -1:
                continue
            if p < -1 or p >= P:
                err |= ERR_RANGE
                continue
            if rrow(p) is None:
                err |= ERR_RANGE
                continue
            if rrow(p) >= 0 and m != "resident_dup_checked":
                continue
            if p in seen and m != "no_dup_check" and (not union or m == "union_repeat_is_error"):
                err |= ERR_DUP
            seen.add(p)
        if newest < -1 or newest >= P:
            err |= ERR_RANGE
        if err:
            return [-1] * k, [], err
        out, hits, misses = [None] * k, [], []
        first = {}
        for i in order:
            p = sel[i]
            if union and p != -1 and p in first and m != "union_counts_repeats":
                continue
            first.setdefault(p, i)
            hot = p in self.page_table
            if p == -1:
                out[i] = -1
            elif m == "resident_after_hot" and hot:
                out[i] = self.page_table[p]
                hits.append(out[i])
            elif m == "resident_after_newest" and newest >= 0 and p == newest:
                out[i] = B
            elif rrow(p) >= 0:
                out[i] = B + 1 + rrow(p)
                if m == "resident_is_hit" and hot:
                    hits.append(self.page_table[p])
                if m == "resident_counts_miss":
                    misses.append(i)
            elif newest >= 0 and p == newest and m != "newest_is_miss":
                out[i] = B
            elif hot:
                out[i] = self.page_table[p]
                hits.append(out[i])
            else:
                misses.append(i)
        misses.sort()
        ev = [s for s in self.lru if s not in hits]
        if m == "victims_from_newest_end":
            ev = ev[::-1]
        M = len(misses)
        plan = []
        for j, i in enumerate(misses):
            s = ev[j]
            p = sel[i]
            old = self.slot_pos[s]
            if old >= 0 and m != "keep_stale_mapping":
                del self.page_table[old]
            self.slot_pos[s] = p
            self.page_table[p] = s
            if self.host is not None and not skip_io and m != "no_fetch":
                self.hot[s] = self.host(p + 1 if m == "fetch_off_by_one" else p)
            out[i] = s
            plan.append((p, s))
        for i, p in enumerate(sel):
            if out[i] is None:
                out[i] = out[first[p]]
        hs = sorted(hits)
        if m == "hits_in_selection_order":
            hs = hits
        if m == "hits_before_misses":
            self.lru = ev[M:] + hs + ev[:M]
        elif m == "misses_oldest":
            self.lru = ev[:M] + ev[M:] + hs
        elif m == "misses_reversed":
            self.lru = ev[M:] + ev[:M][::-1] + hs
        elif m == "victims_from_newest_end":
            self.lru = (ev[M:] + ev[:M])[::-1][::-1]
            self.lru = [s for s in self.lru if s not in hs] + hs
        else:
            self.lru = ev[M:] + ev[:M] + hs
        self.miss_count = M + (1 if m == "count_newest" and newest in sel else 0)
        return out, plan, 0


MUTATIONS = ["no_dup_check", "newest_is_miss", "victims_from_newest_end", "keep_stale_mapping",
             "no_fetch", "fetch_off_by_one", "hits_in_selection_order", "hits_before_misses",
             "misses_oldest", "misses_reversed", "count_newest",
             # resident tier
             "resident_after_hot", "resident_after_newest", "resident_is_hit",
             "resident_counts_miss", "resident_no_offset", "resident_no_entry_check",
             "resident_dup_checked",
             # union mode
             "union_last_reference", "union_counts_repeats", "union_repeat_is_error"]


@pytest.mark.parametrize("mutation", MUTATIONS)
def test_planted_mistake_is_caught(mutation):
    cls = type("M_" + mutation, (_Mutant,), {"mutation": mutation})
    failed = []
    for pin in ALL_PINS:
        try:
            pin(cls)
        except (AssertionError, KeyError, IndexError, TypeError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"no pin catches the planted mistake {mutation!r}"


def test_unmutated_copy_passes_every_pin():
    cls = type("M_none", (_Mutant,), {"mutation": None})
    for pin in ALL_PINS:
        pin(cls)


# ---------------------------------------------------------------------- #
# Block-id selections                                                      #
# ---------------------------------------------------------------------- #
def test_expand_blocks_written_out():
    from oracle.tiny import expand_blocks
    assert expand_blocks([3, -1, 0], 4) == [12, 13, 14, 15, -1, -1, -1, -1, 0, 1, 2, 3]
    assert expand_blocks([5, 2], 1) == [5, 2]
    assert expand_blocks([], 4) == []
    bad = expand_blocks([-2], 2)
    assert all(p < -1 for p in bad)


def test_block_selection_resolves_like_its_positions():
    """A block-id list resolves exactly as its expanded position list does,
    including the error for a negative block id other than -1."""
    from oracle.tiny import expand_blocks
    u = Unit(16, 64, k=8)
    out, plan, err = u.resolve(expand_blocks([2, 7], 4))
    assert err == 0 and u.miss_count == 8 and sorted(p for p, _ in plan) == list(range(8, 12)) + list(range(28, 32))
    out, plan, err = u.resolve(expand_blocks([7, -3], 4))
    assert err == ERR_RANGE and out == [-1] * 8


# ---------------------------------------------------------------------- #
# Admission with preload (reading R16)                                     #
# ---------------------------------------------------------------------- #
@pytest.mark.parametrize("k", [1, 3, 8])
def test_admit_closed_form(k):
    """Preloading n positions: slot s holds position s, LRU = empties then the
    preloaded slots, bytes equal the host rows -- for any list length used to
    get there; n = 0 is the reset state."""
    B, P = 8, 20
    host = lambda p: bytes([p] * 4)  # noqa: E731
    for n in range(0, B + 1):
        u = Unit(B, P, k=k, host=host)
        u.resolve([5] + [-1] * (k - 1))               # some prior state
        plan = u.admit(n, k=k)
        assert u.slot_pos == list(range(n)) + [-1] * (B - n)
        assert u.lru == list(range(n, B)) + list(range(n))
        assert u.page_table == {s: s for s in range(n)} and u.miss_count == 0
        assert [u.hot[s] for s in range(n)] == [host(s) for s in range(n)]
        assert sorted(plan) == [(s, s) for s in range(n)]


def test_admit_c_equals_python():
    from oracle.coracle import OracleLayer
    R, k, B, P, rec = 3, 4, 12, 40, 8
    host = np.random.default_rng(3).integers(0, 256, size=(R, P, rec), dtype=np.uint8)
    c = OracleLayer(R, k, B, P, rec, host=host)
    c.reset()
    c.resolve(np.array([[1, 2, 3, 4]] * R, np.int32))
    for r, n in enumerate([0, 7, 12]):
        c.admit(r, n)
        u = Unit(B, P, k=k, host=lambda p, r=r: bytes(host[r, p]))
        u.admit(n, k=k)
        assert list(c.slot_pos[r]) == u.slot_pos and list(c.lru[r]) == u.lru
        assert c.miss_count[r] == 0
        for s in range(n):
            assert bytes(c.hot[r, s]) == u.hot[s]


def test_strided_host_rows_give_the_same_result():
    """The C model reads host row p at req_stride*r + row_stride*p: a pool
    whose rows are interleaved with another layer's gives the same state and
    bytes as a contiguous copy of the same rows."""
    from oracle.coracle import OracleLayer
    R, k, B, P, rec = 2, 5, 9, 30, 16
    rng = np.random.default_rng(11)
    big = rng.integers(0, 256, size=(R, P, 3, rec), dtype=np.uint8)
    strided = big[:, :, 1, :]                 # rows 48 bytes apart
    flat = np.ascontiguousarray(strided)
    a = OracleLayer(R, k, B, P, rec, host=strided)
    b = OracleLayer(R, k, B, P, rec, host=flat)
    a.reset(); b.reset()
    for t in range(10):
        sel = np.stack([rng.choice(P, size=k, replace=False) for _ in range(R)]).astype(np.int32)
        oa, _ = a.resolve(sel)
        ob, _ = b.resolve(sel)
        np.testing.assert_array_equal(oa, ob)
        np.testing.assert_array_equal(a.hot, b.hot)
    for r in range(R):
        for s in range(B):
            p = a.slot_pos[r, s]
            if p >= 0:
                assert bytes(a.hot[r, s]) == bytes(flat[r, p])


def _preload_matches_replay(preload):
    """Whether ``preload(layer, r, n)`` gives a shared-index layer the bytes
    that replaying the anchor's admission plan into it gives, for several n
    (rows above the prefill split included, up to the whole buffer)."""
    from oracle.coracle import OracleLayer
    k, B, P, split, rec = 4, 16, 40, 10, 8
    rng = np.random.default_rng(21)
    host_a = rng.integers(0, 256, size=(1, split, rec), dtype=np.uint8)
    host_f = rng.integers(0, 256, size=(1, split, rec), dtype=np.uint8)
    for n in (0, 1, 7, 10, 13, 16):
        f1 = OracleLayer(1, k, B, P, rec, host=host_f, host_split=split, metadata=False)
        f2 = OracleLayer(1, k, B, P, rec, host=host_f, host_split=split, metadata=False)
        tail = rng.integers(0, 256, size=f1.host_tail[0].shape, dtype=np.uint8)
        for f in (f1, f2):   # the same written-back tail rows, and stale hot rows
            f.host_tail[0] = tail
            f.hot[0] = 0x5C
        preload(f1, 0, n)
        a = OracleLayer(1, k, B, P, rec, host=host_a, host_split=split)
        a.reset()
        for c0 in range(0, n, k):   # the admission's consecutive lists of k positions
            chunk = np.full((1, k), -1, np.int32)
            m = min(n, c0 + k) - c0
            chunk[0, :m] = np.arange(c0, c0 + m)
            _, e = a.resolve(chunk)
            assert e == 0
            a.replay_into(f2)
        if not np.array_equal(f1.hot, f2.hot):
            return False
        for s in range(n):             # slot s holds the shared layer's own row s
            exp = host_f[0, s] if s < split else tail[s - split]
            if not np.array_equal(f1.hot[0, s], exp):
                return False
    return True


def test_shared_layer_preload_equals_replay_of_the_admission_plan():
    """A shared-index layer's side of an admission (``preload_bytes``) holds
    exactly the bytes that replaying the anchor's admission plan into it
    gives (gentlecold.top §3.6: a shared layer keeps its slots in lockstep
    with its anchor and takes the bytes of the anchor's plan from its own host
    pool), including rows above the prefill split, which come from the
    layer's own written-back tail."""
    from oracle.coracle import OracleLayer
    assert _preload_matches_replay(OracleLayer.preload_bytes)


def _preload_off_by_one(o, r, n):
    for s in range(n):
        o.hot[r, s] = o.host_row(r, min(s + 1, o.P - 1))


def _preload_ignores_split(o, r, n):
    for s in range(n):
        o.hot[r, s] = o._host_keep[r, min(s, o.host_split - 1)]


def _preload_one_short(o, r, n):
    for s in range(max(0, n - 1)):
        o.hot[r, s] = o.host_row(r, s)


@pytest.mark.parametrize("mutant", [_preload_off_by_one, _preload_ignores_split,
                                    _preload_one_short])
def test_preload_pin_catches_planted_mistakes(mutant):
    assert not _preload_matches_replay(mutant)


# ---------------------------------------------------------------------- #
# Short requests (reading R17)                                             #
# ---------------------------------------------------------------------- #
import copy  # noqa: E402


def _short_run(cls, B=16, k=5, n=6, steps=9, seed=0, check=True):
    """A request admitted with n positions preloaded, then decoded on the
    short path until seq_len reaches B: every step writes the previous token
    back (the host callable returns what the write-back stored), grows the
    buffer by it and looks the selection up.  With ``check``, asserts the
    closed forms after every step; returns False on the first failure."""
    rng = random.Random(seed)
    store = {}
    host = lambda p: store.get(p, ("prefill", p))   # noqa: E731
    u = cls(B, 4 * B, k=k, host=host)
    u.admit(n, k=k)
    t = 0
    while n + t + 1 <= B and t < steps:
        newest = n + t
        prev = newest - 1 if t > 0 else -1
        seq_len = n + t + 1
        if prev >= 0:
            store[prev] = ("written", prev)     # the write-back of the previous token
        pool = list(range(seq_len))
        sel = rng.sample(pool, min(k - 1, seq_len)) + [-1]
        rng.shuffle(sel)
        ref = copy.deepcopy(u)
        out, plan, err = u.resolve_short(sel, newest, seq_len, prev=prev)
        ok = err == 0
        grown = n + t                           # slots 0..grown-1 hold their positions
        ok = ok and u.slot_pos[:grown] == list(range(grown))
        ok = ok and all(u.hot[s] == host(s) for s in range(grown))
        ok = ok and u.lru == list(range(grown, B)) + list(range(n)) + list(range(n, grown))
        ok = ok and plan == ([(prev, prev)] if prev >= 0 else [])
        # the general resolve on the grown state gives the same slots, all hits
        if prev >= 0:
            ref.resolve([prev])
        o2, p2, e2 = ref.resolve(sel, newest)
        ok = ok and out == o2 and p2 == [] and e2 == 0
        if check:
            assert ok, f"step {t}"
        elif not ok:
            return False
        t += 1
    return True


@pytest.mark.parametrize("B,k,n", [(16, 5, 6), (8, 3, 0), (32, 7, 31), (12, 12, 1)])
def test_short_path_grows_in_order_and_equals_the_general_resolve(B, k, n):
    """Closed forms of R17 for an admitted short request: slot s holds
    position s and its record, the LRU order is the remaining empties, the
    preloaded slots, then the grown ones, each growth is one planned miss into
    the next empty slot, and every lookup equals the general resolve's output
    on the same state (all hits, no misses)."""
    for seed in range(4):
        _short_run(Unit, B=B, k=k, n=n, steps=B, seed=seed)


def _short_error_pin(cls):
    """A position at or past seq_len, or a bad newest position, fails the
    lookup (all -1) after the growth has happened; a repeated position is not
    an error; padding stays -1; a resident row comes first."""
    u = cls(8, 40, k=4, host=lambda p: p)
    u.admit(3, k=4)
    out, plan, err = u.resolve_short([0, 1, 4, -1], 3, 4, prev=-1)
    assert err == ERR_RANGE and out == [-1] * 4 and plan == []
    out, plan, err = u.resolve_short([0, 0, 2, -1], 4, 5, prev=3)
    assert err == 0 and out == [0, 0, 2, -1] and plan == [(3, 3)] and u.slot_pos[3] == 3
    out, plan, err = u.resolve_short([0, 1, 2, 4], 4, 5, prev=-1)
    assert err == 0 and out == [0, 1, 2, 8] and u.miss_count == 0
    out, plan, err = u.resolve_short([0, 1, 2, 3], 40, 5)
    assert err == ERR_RANGE and out == [-1] * 4
    out, plan, err = u.resolve_short([0, 9, 2, -1], 4, 5, res_blocks=[-1, -1, 7], res_tok=4)
    assert err == 0 and out == [0, 8 + 1 + 7 * 4 + 1, 2, -1]


def test_short_path_errors_and_repeats():
    _short_error_pin(Unit)


def test_short_to_long_transition():
    """At seq_len = B + 1 the general resolve takes over: the token at B - 1
    was never grown (its step is no longer short), so it is host-only, misses
    and takes the one empty slot, B - 1, which the growths left least recent."""
    B, k, n = 8, 3, 5
    store = {}
    u = Unit(B, 40, k=k, host=lambda p: store.get(p, p))
    u.admit(n, k=k)
    for t in range(1, B - n):                 # grow positions n .. B-2
        store[n + t - 1] = ("w", n + t - 1)
        u.resolve_short([0, -1, -1], n + t, n + t + 1, prev=n + t - 1)
    assert u.slot_pos == list(range(B - 1)) + [-1]
    assert u.lru == [B - 1] + list(range(B - 1))
    store[B - 1] = ("w", B - 1)                 # the transition step's write-back
    out, plan, err = u.resolve([B - 1, 0, B], newest=B)
    assert err == 0 and out == [B - 1, 0, B] and plan == [(B - 1, B - 1)]
    assert u.hot[B - 1] == ("w", B - 1) and u.lru == list(range(1, B - 1)) + [B - 1, 0]


def test_short_path_python_equals_c():
    """The C model's step with per-request sequence lengths (short requests
    grown and looked up by position, long ones resolved) equals the Python
    model's, field by field, over mixed batches, a resident table included."""
    from oracle.coracle import OracleLayer
    R, k, B, P, rec = 4, 6, 16, 64, 8
    rng = np.random.default_rng(5)
    host = rng.integers(0, 256, size=(R, P, rec), dtype=np.uint8)
    lens0 = [3, 10, 20, 40]                     # two short, two long
    c = OracleLayer(R, k, B, P, rec, host=host)
    c.reset()
    py = []
    for r in range(R):
        u = Unit(B, P, k=k, host=lambda p, r=r: bytes(host[r, p]))
        pre = lens0[r] if lens0[r] <= B else 0
        u.admit(pre, k=k)
        c.admit(r, pre)
        py.append(u)
    blocks = np.full((R, P // 8), -1, np.int32)
    blocks[2, 1] = 3
    for t in range(8):
        seq = np.array([L + t + 1 for L in lens0], np.int32)
        newest = seq - 1
        prev = np.where(np.full(R, t > 0), newest - 1, -1).astype(np.int32)
        sel = np.full((R, k), -1, np.int32)
        for r in range(R):
            m = min(k - 1, int(seq[r]))
            sel[r, :m] = rng.choice(int(seq[r]), size=m, replace=False)
        out, err = c.resolve_with_seq_lens(sel, newest, prev, seq, res_blocks=blocks, res_tok=8)
        for r in range(R):
            u = py[r]
            if seq[r] <= B:
                o, plan, e = u.resolve_short(sel[r].tolist(), int(newest[r]), int(seq[r]),
                                             prev=int(prev[r]), res_blocks=blocks[r].tolist(),
                                             res_tok=8)
            else:
                o, plan, e = u.resolve(sel[r].tolist(), int(newest[r]),
                                       res_blocks=blocks[r].tolist(), res_tok=8)
            assert out[r].tolist() == o and c.unit_err[r] == e
            assert c.slot_pos[r].tolist() == u.slot_pos and c.lru[r].tolist() == u.lru
            assert int(c.miss_count[r]) == u.miss_count
            assert list(zip(c.plan_pos[r, :c.plan_count[r]].tolist(),
                            c.plan_slot[r, :c.plan_count[r]].tolist())) == plan
            for s in range(B):
                if u.slot_pos[s] >= 0:
                    assert bytes(c.hot[r, s]) == u.hot[s]


class _ShortNoNewest(Unit):
    def resolve_short(self, sel, newest, seq_len, prev=-1, res_blocks=None, res_tok=1):
        return super().resolve_short(sel, -1 if newest < seq_len - 1 else -1, seq_len + 1,
                                     prev, res_blocks, res_tok)


class _ShortRangeOffByOne(Unit):
    def resolve_short(self, sel, newest, seq_len, prev=-1, res_blocks=None, res_tok=1):
        return super().resolve_short([p if p < seq_len + 1 else p for p in sel], newest,
                                     seq_len + 1, prev, res_blocks, res_tok)


class _ShortGrowsIntoRecentSlot(Unit):
    def resolve_short(self, sel, newest, seq_len, prev=-1, res_blocks=None, res_tok=1):
        if prev >= 0 and prev not in self.page_table:
            self.lru = self.lru[::-1]           # the victim becomes the most recent slot
            out = super().resolve_short(sel, newest, seq_len, prev, res_blocks, res_tok)
            return out
        return super().resolve_short(sel, newest, seq_len, prev, res_blocks, res_tok)


class _ShortNoGrowth(Unit):
    def resolve_short(self, sel, newest, seq_len, prev=-1, res_blocks=None, res_tok=1):
        return super().resolve_short(sel, newest, seq_len, -1, res_blocks, res_tok)


@pytest.mark.parametrize("cls", [_ShortNoNewest, _ShortGrowsIntoRecentSlot, _ShortNoGrowth])
def test_short_path_pins_catch_planted_mistakes(cls):
    caught = not all(_short_run(cls, B=16, k=5, n=6, steps=16, seed=s, check=False)
                     for s in range(4))
    assert caught


def test_short_path_range_pin_catches_an_off_by_one():
    with pytest.raises(AssertionError):
        _short_error_pin(_ShortRangeOffByOne)
