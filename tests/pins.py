"""Pins for the oracle: checks that tie it to the pages and to mathematics.

Each ``pin_*`` takes a unit class with the API of ``oracle.tiny.Unit``
(``Unit(B, P, k=None, host=None)``, ``resolve(sel, newest) -> (out, plan,
err)``, fields ``slot_pos``, ``lru``, ``page_table``, ``miss_count``, ``hot``)
and raises ``AssertionError`` when the unit disagrees with the pin.  The same
pins run on the Python model, on the C model (through ``CUnit``) and on planted
mistakes (``test_oracle_pins.py``), which must each fail at least one pin.
"""
import os
import random

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------------- #
def parse_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            rows.append((key, rest))
    return rows


def _ints(s):
    return [int(x) for x in s.split()]


# ---------------------------------------------------------------------- #
# C model adapter with the Python model's API                            #
# ---------------------------------------------------------------------- #
class CUnit:
    """One unit of the C oracle behind the ``oracle.tiny.Unit`` API."""

    def __init__(self, B, P, k=None, host=None):
        from oracle.coracle import OracleLayer
        self.B, self.P = B, P
        self.k = k
        self._host = host
        self._L = None

    def _layer(self, k):
        if self._L is None:
            from oracle.coracle import OracleLayer
            rec = 8
            host = None
            if self._host is not None:
                host = np.zeros((1, self.P, rec), np.uint8)
                for p in range(self.P):
                    host[0, p] = np.frombuffer(self._host(p), np.uint8)
            self._L = OracleLayer(1, k, self.B, self.P, rec, host=host,
                                  keep_bytes=self._host is not None)
            self._L.reset()
            if self._pending is not None:
                sp, lru = self._pending
                self._L.slot_pos[0] = sp
                self._L.lru[0] = lru
                for s, p in enumerate(sp):
                    if p >= 0:
                        self._L.page_table[0, p] = s
        return self._L

    _pending = None

    # state preset before the first resolve (used by the worked example)
    def preset(self, slot_pos, lru):
        self._pending = (list(slot_pos), list(lru))

    def resolve(self, sel, newest=-1, skip_io=False, res_blocks=None, res_tok=1, union=False):
        L = self._layer(len(sel))
        rb = None if res_blocks is None else np.array([res_blocks], np.int32)
        out, e = L.resolve(np.array([sel], np.int32), np.array([newest], np.int32),
                           io=not skip_io, res_blocks=rb, res_tok=res_tok, union=union)
        plan = [(int(L.plan_pos[0, j]), int(L.plan_slot[0, j])) for j in range(L.plan_count[0])]
        return [int(x) for x in out[0]], plan, int(e)

    @property
    def slot_pos(self):
        return [int(x) for x in self._layer(self.k or 1).slot_pos[0]]

    @property
    def lru(self):
        return [int(x) for x in self._layer(self.k or 1).lru[0]]

    @property
    def page_table(self):
        pt = self._layer(self.k or 1).page_table[0]
        return {int(p): int(pt[p]) for p in np.flatnonzero(pt >= 0)}

    @property
    def miss_count(self):
        return int(self._layer(self.k or 1).miss_count[0])

    @property
    def hot(self):
        L = self._layer(self.k or 1)
        return [bytes(L.hot[0, s]) for s in range(self.B + 1)]


def make(cls, B, P, k=None, host=None, slot_pos=None, lru=None):
    u = cls(B, P, k=k, host=host)
    if slot_pos is not None:
        if hasattr(u, "preset"):
            u.preset(slot_pos, lru)
        else:
            u.slot_pos = list(slot_pos)
            u.lru = list(lru)
            u.page_table = {p: s for s, p in enumerate(slot_pos) if p >= 0}
    return u


# ---------------------------------------------------------------------- #
def pin_example_b(cls):
    """gentlecold.top deep dive §3.5 worked example: exact slots and LRU."""
    g = dict(parse_golden("example_b_resolve.txt"))
    B, k = int(g["B"]), int(g["k"])
    u = make(cls, B, 64, k=k, slot_pos=_ints(g["slot_pos"]), lru=_ints(g["lru"]))
    out, plan, err = u.resolve(_ints(g["sel"]), newest=int(g["newest"]))
    assert err == 0
    assert out == _ints(g["expect_out"]), out
    assert list(u.lru) == _ints(g["expect_lru"]), u.lru
    assert list(u.slot_pos) == _ints(g["expect_slot_pos"]), u.slot_pos
    assert u.miss_count == int(g["expect_misses"])
    exp_plan = [tuple(int(x) for x in e.split(":")) for e in g["expect_plan"].split()]
    assert [tuple(p) for p in plan] == exp_plan
    pt = u.page_table
    assert pt.get(25) == 0 and pt.get(12) == 2 and pt.get(16) == 6 and 10 not in pt
    assert 30 not in pt  # the newest token is not in the LRU page table


def pin_example_a(cls):
    """notes.kuangjux.top §5 capacity example: miss counts and evictions."""
    rows = parse_golden("example_a_capacity.txt")
    steps = [_ints(v) for key, v in rows if key == "step"]
    k = int(dict(rows)["k"])
    caps = {}
    for key, v in rows:
        if key == "capacity":
            cap, _, m = v.partition(":")
            caps[int(cap)] = _ints(m)
    evicted = {}
    for key, v in rows:
        if key == "evicted":
            cap, _, m = v.partition(":")
            step, pos = _ints(m)
            evicted.setdefault(int(cap), {})[step] = pos
    for cap, exp in caps.items():
        u = make(cls, cap, 16, k=k)
        got, before = [], set()
        for t, s in enumerate(steps, start=1):
            before = {p for p in u.slot_pos if p >= 0}
            out, plan, err = u.resolve(list(s))
            assert err == 0
            got.append(u.miss_count)
            after = {p for p in u.slot_pos if p >= 0}
            if cap in evicted and t in evicted[cap]:
                assert before - after == {evicted[cap][t]}, (cap, t, before, after)
        assert got == exp, (cap, got, exp)


def textbook_lru(refs, frames):
    """Classic single-page LRU (a list, most recent at the end): per-step hit flags."""
    mem, hits = [], []
    for p in refs:
        if p in mem:
            mem.remove(p)
            mem.append(p)
            hits.append(True)
        else:
            if len(mem) == frames:
                mem.pop(0)
            mem.append(p)
            hits.append(False)
    return hits, set(mem)


def pin_textbook_lru(cls, seeds=range(6)):
    """k = 1 reduces to the textbook LRU page-replacement algorithm."""
    # Silberschatz et al., Operating System Concepts, LRU example: 12 faults.
    refs = [7, 0, 1, 2, 0, 3, 0, 4, 2, 3, 0, 3, 2, 1, 2, 0, 1, 7, 0, 1]
    u = make(cls, 3, 8, k=1)
    faults = 0
    for p in refs:
        u.resolve([p])
        faults += u.miss_count
    assert faults == 12, faults
    for seed in seeds:
        rnd = random.Random(seed)
        frames = rnd.choice([1, 2, 3, 5])
        refs = [rnd.randrange(9) for _ in range(40)]
        exp_hits, exp_res = textbook_lru(refs, frames)
        u = make(cls, frames, 9, k=1)
        for t, p in enumerate(refs):
            u.resolve([p])
            assert (u.miss_count == 0) == exp_hits[t], (seed, t)
        assert {p for p in u.slot_pos if p >= 0} == exp_res


def pin_hit_order(cls):
    """Reading R1: among hits of one step, the lowest slot is evicted first.

    Fill slots 0..3 with positions 0..3, then select them in the order
    3, 2, 1, 0 (selection order opposite to slot order) plus one new position
    so that all four are this step's hits.  Later steps with fresh positions
    must then evict them slot 0 first, then 1, 2, 3.
    """
    u = make(cls, 5, 64, k=5)
    u.resolve([0, 1, 2, 3, -1])             # slots 0..3 <- positions 0..3
    u.resolve([3, 2, 1, 0, 10])             # all four hit; 10 -> slot 4
    order = []
    for t in range(4):
        before = {p: s for s, p in enumerate(u.slot_pos) if p >= 0}
        u.resolve([20 + t, -1, -1, -1, -1])
        after = {p for p in u.slot_pos if p >= 0}
        gone = set(before) - after
        assert len(gone) == 1
        order.append(before[gone.pop()])
    # slot 4 (position 10, fetched in the step where the others hit) goes first,
    # then the hits by ascending slot.
    assert order == [4, 0, 1, 2], order


def pin_miss_order(cls):
    """Reading R2: the j-th miss takes the j-th oldest evictable; earlier list
    index = older among this step's fetches."""
    u = make(cls, 4, 64, k=4)
    out, plan, _ = u.resolve([7, 5, 9, -1])
    assert out[:3] == [0, 1, 2] and out[3] == -1
    assert list(u.lru) == [3, 0, 1, 2]
    out, plan, _ = u.resolve([40, 41, -1, -1])
    assert out[:2] == [3, 0]                 # oldest evictables, in list order
    assert list(u.lru) == [1, 2, 3, 0]


def pin_newest_and_padding(cls):
    """Reading R4/R6/R8: newest -> row B, not a miss; -1 -> -1, not a miss."""
    u = make(cls, 4, 64, k=4)
    out, plan, err = u.resolve([9, -1, 33, 5], newest=33)
    assert err == 0
    assert out[1] == -1 and out[2] == 4
    assert u.miss_count == 2
    assert 33 not in {p for p in u.slot_pos}


def pin_errors(cls):
    """Reading R6: duplicates / out-of-range fail the unit, state untouched."""
    u = make(cls, 4, 16, k=3)
    u.resolve([1, 2, 3])
    snap = (list(u.slot_pos), list(u.lru), dict(u.page_table))
    out, plan, err = u.resolve([4, 4, 5])
    assert err == 2 and out == [-1, -1, -1] and plan == []
    assert (list(u.slot_pos), list(u.lru), dict(u.page_table)) == snap
    out, plan, err = u.resolve([4, 16, 5])
    assert err == 1 and out == [-1, -1, -1]
    out, plan, err = u.resolve([4, -7, 5])
    assert err == 1
    out, plan, err = u.resolve([4, 6, 5], newest=99)
    assert err == 1
    assert (list(u.slot_pos), list(u.lru), dict(u.page_table)) == snap


def pin_invariants(cls, seeds=range(25)):
    """Structure invariants after every step on random small traces, plus
    cold-start and steady-state closed forms and the bytes invariant."""
    for seed in seeds:
        rnd = random.Random(1000 + seed)
        k = rnd.randint(1, 6)
        B = k + rnd.randint(0, 4)
        P = rnd.randint(k + 2, 24)
        host = lambda p: bytes([(p * 37 + i) & 0xFF for i in range(8)])  # noqa: E731
        u = make(cls, B, P, k=k, host=host)
        for t in range(12):
            nsel = rnd.randint(0, k)
            S = rnd.sample(range(P), nsel)
            sel = S + [-1] * (k - nsel)
            rnd.shuffle(sel)
            newest = rnd.choice([-1] + S) if S and rnd.random() < 0.3 else -1
            res_before = {p for p in u.slot_pos if p >= 0}
            out, plan, err = u.resolve(sel, newest=newest)
            assert err == 0
            exp_m = sum(1 for p in sel if p != -1 and p != newest and p not in res_before)
            assert u.miss_count == exp_m
            if t == 0:
                assert u.miss_count == sum(1 for p in sel if p not in (-1, newest))
            slot_pos, lru, pt = list(u.slot_pos), list(u.lru), dict(u.page_table)
            assert sorted(lru) == list(range(B))
            for p, s in pt.items():
                assert slot_pos[s] == p
            assert len(pt) == sum(1 for p in slot_pos if p >= 0)
            used = [o for o in out if 0 <= o < B]
            assert len(used) == len(set(used))
            for i, p in enumerate(sel):
                if p == -1:
                    assert out[i] == -1
                elif p == newest:
                    assert out[i] == B
                else:
                    assert 0 <= out[i] < B and slot_pos[out[i]] == p
            hot = u.hot
            for s, p in enumerate(slot_pos):
                if p >= 0:
                    assert hot[s] == host(p), (seed, t, s, p)
            # the same selection again: everything hits
        out2, _, _ = u.resolve(sel, newest=newest)
        assert u.miss_count == 0 and out2 == out


def pin_disjoint_at_b_equals_k(cls):
    """Closed form: B = k and disjoint consecutive selections -> M = k each step."""
    k = 4
    u = make(cls, k, 64, k=k)
    for t in range(6):
        u.resolve([t * k + i for i in range(k)])
        assert u.miss_count == k


def pin_belady_bound(cls, seeds=range(40)):
    """LRU never beats the offline optimum (brute force on tiny traces)."""
    from oracle.tiny import optimal_misses
    for seed in seeds:
        rnd = random.Random(5000 + seed)
        B = rnd.randint(1, 4)
        k = rnd.randint(1, B)
        steps = rnd.randint(2, 6)
        trace = [rnd.sample(range(8), rnd.randint(1, k)) for _ in range(steps)]
        u = make(cls, B, 8, k=k)
        total = 0
        for s in trace:
            u.resolve(list(s) + [-1] * (k - len(s)))
            total += u.miss_count
        assert total >= optimal_misses(trace, B), (seed, total)


# ---------------------------------------------------------------------- #
# The resident tier (docs.vllm.ai "HiSparse local KV offload architecture", #
# "Hot lookup and LRU": resident page -> resident physical row, before the  #
# hot lookup; resident hits bypass the hot LRU and host copies)             #
# ---------------------------------------------------------------------- #
def _snap(u):
    return list(u.slot_pos), list(u.lru), dict(u.page_table), u.miss_count


def pin_resident_none_is_plain(cls, seeds=range(8)):
    """An all -1 block table changes nothing: same outputs, plan and state."""
    for seed in seeds:
        rnd = random.Random(7000 + seed)
        k, B, P, tok = 5, 8, 40, 4
        a, b = make(cls, B, P, k=k), make(cls, B, P, k=k)
        blocks = [-1] * (P // tok)
        for _ in range(10):
            sel = rnd.sample(range(P), k)
            newest = rnd.choice([-1, sel[0]])
            ra = a.resolve(sel, newest=newest, res_blocks=blocks, res_tok=tok)
            rb = b.resolve(sel, newest=newest)
            assert ra == rb and _snap(a) == _snap(b)


def pin_resident_masks(cls, seeds=range(20)):
    """A resident selection acts on the cache exactly as padding would, and
    outputs B + 1 + (entry * block size + offset): the state, plan and miss
    count equal those of the same list with its resident entries set to -1.
    Block tables change from step to step, so positions resident now are
    often hot from earlier steps, and the newest position is sometimes
    resident (the resident check comes first)."""
    for seed in seeds:
        rnd = random.Random(8000 + seed)
        k = rnd.randint(2, 6)
        B = k + rnd.randint(0, 3)
        tok = rnd.choice([1, 2, 4])
        P = tok * rnd.randint(8, 12)
        host = lambda p: bytes([(p * 11 + i) & 0xFF for i in range(8)])  # noqa: E731
        a, b = make(cls, B, P, k=k, host=host), make(cls, B, P, k=k, host=host)
        for t in range(12):
            nb = P // tok
            blocks = [rnd.randrange(50) if rnd.random() < 0.35 else -1 for _ in range(nb - 1)]
            sel = rnd.sample(range(P), rnd.randint(1, k))
            sel += [-1] * (k - len(sel))
            rnd.shuffle(sel)
            newest = rnd.choice([-1] + [p for p in sel if p >= 0])
            row = {}
            for p in sel:
                if p >= 0 and p // tok < len(blocks) and blocks[p // tok] >= 0:
                    row[p] = blocks[p // tok] * tok + p % tok
            masked = [-1 if p in row else p for p in sel]
            oa, pa, ea = a.resolve(sel, newest=newest, res_blocks=blocks, res_tok=tok)
            ob, pb, eb = b.resolve(masked, newest=newest)
            assert ea == 0 and eb == 0
            assert [tuple(x) for x in pa] == [tuple(x) for x in pb]
            assert _snap(a) == _snap(b), (seed, t)
            for i, p in enumerate(sel):
                assert oa[i] == (B + 1 + row[p] if p in row else ob[i]), (seed, t, i)
            assert a.hot[:B] == b.hot[:B]


def pin_resident_all(cls):
    """A request whose every selection is resident leaves its cache untouched."""
    k, B, P, tok = 4, 6, 32, 8
    u = make(cls, B, P, k=k)
    u.resolve([1, 9, 17, 25])
    snap = _snap(u)[:3]
    blocks = [3, 0, 5, 2]
    out, plan, err = u.resolve([9, 2, 30, -1], newest=30, res_blocks=blocks, res_tok=tok)
    assert err == 0 and plan == [] and u.miss_count == 0
    assert out == [B + 1 + 0 * 8 + 1, B + 1 + 3 * 8 + 2, B + 1 + 2 * 8 + 6, -1]
    assert _snap(u)[:3] == snap


def pin_resident_errors(cls):
    """An invalid block entry (below -1) or a row past int32 fails the unit,
    state untouched, but only when a selected position falls in that block."""
    k, B, P, tok = 3, 4, 16, 4
    u = make(cls, B, P, k=k)
    u.resolve([1, 2, 3])
    snap = _snap(u)[:3]
    out, plan, err = u.resolve([4, 9, 0], res_blocks=[-1, -5, 2, -1], res_tok=tok)
    assert err == 1 and out == [-1] * 3 and _snap(u)[:3] == snap
    out, plan, err = u.resolve([4, 9, 0], res_blocks=[-1, 2**29, 2, -1], res_tok=tok)
    assert err == 1 and out == [-1] * 3 and _snap(u)[:3] == snap
    out, plan, err = u.resolve([0, 9, 13], res_blocks=[-1, -1, 2, -5], res_tok=tok)
    assert err == 1
    out, plan, err = u.resolve([0, 9, 1], res_blocks=[-1, -1, 2, -5], res_tok=tok)
    assert err == 0 and out[1] == B + 1 + 2 * 4 + 1


def pin_resident_repeat(cls):
    """A repeated resident position is not a duplicate (it never reaches the
    hot tier) and outputs its row at each index; a repeat that reaches the hot
    tier still fails the unit."""
    k, B, P, tok = 4, 6, 32, 4
    u = make(cls, B, P, k=k)
    out, plan, err = u.resolve([5, 9, 5, 20], res_blocks=[-1, 7, -1, -1], res_tok=tok)
    assert err == 0 and out[0] == out[2] == B + 1 + 7 * 4 + 1 and u.miss_count == 2
    out, plan, err = u.resolve([5, 9, 9, 20], res_blocks=[-1, 7, -1, -1], res_tok=tok)
    assert err == 2 and out == [-1] * 4


RESIDENT_PINS = [pin_resident_none_is_plain, pin_resident_masks, pin_resident_all,
                 pin_resident_errors, pin_resident_repeat]


# ---------------------------------------------------------------------- #
# Union mode: speculative verify rows resolved as one list               #
# (gentlecold.top §6.5: the union of all verify rows' top-k; misses in     #
# (row, top-k) first-reference order)                                     #
# ---------------------------------------------------------------------- #
def pin_union_without_repeats_is_plain(cls, seeds=range(6)):
    for seed in seeds:
        rnd = random.Random(9000 + seed)
        k, B, P = 6, 10, 40
        a, b = make(cls, B, P, k=k), make(cls, B, P, k=k)
        for _ in range(8):
            sel = rnd.sample(range(P), rnd.randint(0, k))
            sel += [-1] * (k - len(sel))
            ra = a.resolve(sel, union=True)
            rb = b.resolve(sel)
            assert ra == rb and _snap(a) == _snap(b)


def pin_union_is_first_reference(cls, seeds=range(20)):
    """Union resolve == resolving the list with every repeat replaced by
    padding, then copying each repeat's output from its first reference
    (state, plan and miss count identical).  Rows overlap like the top-k of
    consecutive draft tokens."""
    for seed in seeds:
        rnd = random.Random(9500 + seed)
        V, kr = rnd.randint(2, 4), rnd.randint(2, 4)
        k, P = V * kr, 30
        B = k + rnd.randint(0, 3)
        host = lambda p: bytes([(p * 13 + i) & 0xFF for i in range(8)])  # noqa: E731
        a, b = make(cls, B, P, k=k, host=host), make(cls, B, P, k=k, host=host)
        base = rnd.sample(range(P), kr)
        for t in range(8):
            rows = []
            for _ in range(V):
                row = [p if rnd.random() < 0.7 else rnd.randrange(P) for p in base]
                row = list(dict.fromkeys(row))          # a top-k row has no repeats
                rows += row + [-1] * (kr - len(row))
            newest = rnd.choice([-1] + [p for p in rows if p >= 0])
            first, masked = {}, []
            for i, p in enumerate(rows):
                if p >= 0 and p in first:
                    masked.append(-1)
                else:
                    first.setdefault(p, i)
                    masked.append(p)
            oa, pa, ea = a.resolve(rows, newest=newest, union=True)
            ob, pb, eb = b.resolve(masked, newest=newest)
            assert ea == 0 and eb == 0
            assert [tuple(x) for x in pa] == [tuple(x) for x in pb]
            assert _snap(a) == _snap(b), (seed, t)
            for i, p in enumerate(rows):
                assert oa[i] == (ob[first[p]] if p >= 0 else -1), (seed, t, i)
            assert a.hot[:B] == b.hot[:B]
            base = [p for p in rows if p >= 0][:kr] or base


def pin_union_example(cls):
    """Two verify rows {1,2,3} and {3,4,1} from the admission state: misses
    1, 2, 3, 4 take slots 0..3 in first-reference order."""
    u = make(cls, 8, 32, k=6)
    out, plan, err = u.resolve([1, 2, 3, 3, 4, 1], union=True)
    assert err == 0 and out == [0, 1, 2, 2, 3, 0]
    assert [tuple(x) for x in plan] == [(1, 0), (2, 1), (3, 2), (4, 3)]
    assert u.miss_count == 4 and list(u.lru) == [4, 5, 6, 7, 0, 1, 2, 3]


UNION_PINS = [pin_union_without_repeats_is_plain, pin_union_is_first_reference,
              pin_union_example]

ALL_PINS = [pin_example_b, pin_example_a, pin_textbook_lru, pin_hit_order, pin_miss_order,
            pin_newest_and_padding, pin_errors, pin_invariants, pin_disjoint_at_b_equals_k,
            pin_belady_bound] + RESIDENT_PINS + UNION_PINS
