"""Pure-Python model of one HiSparse cache unit -- TEST INFRASTRUCTURE ONLY.

A *unit* is one (request, layer) pair.  Units are independent: each keeps its
own slots, LRU order and page table ([P1] §3.3, last paragraph: cross-layer
coordination was dropped, every layer manages its own cache).

State of a unit ([P1] §3.2 and §5.2):
  * ``B`` LRU slots (the hot buffer), plus one extra row with index ``B`` that
    holds the newest token and never takes part in the LRU ([P1] §5.2,
    "newest_slot = HOT_BUFFER_SIZE").
  * ``slot_pos[s]``: the logical position stored in slot ``s`` (-1 = empty).
  * ``lru``: a list of the ``B`` slot ids, oldest first.
  * ``page_table``: ``dict`` logical position -> slot; an absent key means the
    record lives only on the host.
  * ``hot``: the bytes of each slot (only when a host pool is attached).

``resolve`` follows the five stages of the fused kernel ([P1] §3.5) in their
plainest sequential form, with the replacement rule of [P1] §3.3 ("hits of
this step rank as more recent than this step's new misses") and these
readings of points the pages leave open:
  R1  hits of one step are ordered by ascending slot id (the lowest slot is
      evicted first among them);
  R2  misses take victims in selection-list order: the j-th miss takes the
      j-th oldest evictable slot, and among the new fetches an earlier list
      index ends up older;
  R3  empty slots are evictable like any other and keep their LRU place;
  R4  a selection equal to ``newest`` binds to row ``B`` and is a hit that is
      never counted as a miss;
  R6  ``-1`` is padding (output -1); a duplicate or out-of-range position makes
      the whole unit fail with its state untouched and an output row of -1;
  R8  the miss count excludes padding and the newest binding.

With a resident tier (the three-tier resolver of docs.vllm.ai "HiSparse local
KV offload architecture", "Hot lookup and LRU"; gentlecold.top §6.5), a
position whose block has a device-resident copy resolves to that copy before
the hot buffer is consulted, and touches neither the LRU nor the page table:
  R14 the resident check comes first, before the newest binding and the hot
      lookup; a resident selection outputs ``B + 1 + row`` (row = its block's
      entry * block size + the position's offset in the block) and is neither
      a hit nor a miss; a block entry below -1, or a row too large for that
      encoding in int32, fails the unit like an out-of-range position.  The
      duplicate check covers the positions that reach the hot tier: a
      resident position never touches the cache, and the pages place the
      resident exit before the hash table is built, so a repeated resident
      position is not an error and outputs its row at each index.

For speculative verification (gentlecold.top §6.5, "one block resolves the
union of all verify rows' top-k ... misses are allocated in (row, top-k)
first-reference order"; docs.vllm.ai "Hot lookup and LRU", speculative
decoding) a request's verify rows are passed as one list, row after row, in
union mode:
  R15 a position repeated anywhere in the list is resolved once, at its
      first reference, and every later reference outputs the same row; it is
      not an error.  Misses are the first references, in list order; the
      miss count and the plan count each missed position once.

Short requests (gentlecold.top §5.4: when seq_len <= B every token of the
request sits in the buffer in order and the kernel returns slots by position,
with no host IO; the device buffer grows on demand; §5.5: the swap-in
kernel's fast path returns before any LRU work; §5.3: a short request is
admitted with all its tokens preloaded):
  R17 a request whose seq_len (its positions so far, the newest included) is
      at most B takes the short path.  First its buffer grows by the
      previous token: when the step writes a previous token back
      (``prev >= 0``), that token is resolved as a one-entry selection -- a
      miss that takes the least recent slot, or a hit that moves its slot to
      the recent end -- with its miss count and plan (so shared-index layers
      follow); with no previous token the miss count and plan are 0.  Then
      each selection outputs -1 for padding, its resident row when the
      resident table has one, B for the newest token, else the slot numbered
      like its position.  A position outside [0, seq_len), a newest position
      outside [-1, P) or an invalid resident entry fails the lookup (output
      all -1, error code set; the growth has happened).  Repeats are not
      errors: nothing is allocated.  For a request admitted with its first n
      positions preloaded and grown by one token per step since, the least
      recent slot is always the next empty one, so slot s keeps position s
      and the outputs equal those of the general resolve, all hits, without
      its LRU work.  Longer requests are resolved as usual.

See ``tests/test_oracle_pins.py`` for what pins each of these.

[P1] = gentlecold.top, "HiSparse 深度解析：论文、SGLang 实现与 vLLM Hybrid
HiSparse" (sections as numbered on that page).
"""

ERR_RANGE = 1  # a position outside [-1, P), or newest outside [-1, P)
ERR_DUP = 2    # the same position appears twice in one selection
INT32_MAX = 2**31 - 1


class Unit:
    """One (request, layer) cache: B slots + newest row, LRU, page table."""

    def __init__(self, B, P, k=None, host=None):
        if k is not None and B < k:
            raise ValueError("B must be >= k ([P1] §1: B >= k)")
        self.B = B
        self.P = P
        self.slot_pos = [-1] * B
        self.lru = list(range(B))          # oldest first; reset order 0..B-1
        self.page_table = {}               # pos -> slot
        self.host = host                   # callable pos -> bytes, or None
        self.hot = [None] * (B + 1)        # row B = newest slot
        self.miss_count = 0

    # ------------------------------------------------------------------ #
    def resolve(self, sel, newest=-1, skip_io=False, res_blocks=None, res_tok=1, union=False):
        """One RESOLVE of this unit for the selection list ``sel``.

        Returns ``(out, plan, err)``: ``out[i]`` is the physical slot for
        ``sel[i]`` (``B`` for the newest token, -1 for padding, ``B + 1 + row``
        for a resident copy); ``plan`` is the list of ``(pos, slot)`` fetches in
        miss order ([P1] §5.5, the miss plan written where the eviction is
        decided); ``err`` is 0 or a bit-OR of ``ERR_RANGE`` / ``ERR_DUP``.
        ``res_blocks`` (optional) is this request's resident block table: the
        entry of block ``p // res_tok`` is -1 (not resident) or the block's
        index in the resident store (reading R14).  ``union``: repeated
        positions share their first reference's row (reading R15).
        """
        B, P = self.B, self.P
        k = len(sel)

        def resident_row(p):
            if res_blocks is None or p // res_tok >= len(res_blocks):
                return -1
            e = res_blocks[p // res_tok]
            if e < -1:
                return None                # invalid entry
            if e == -1:
                return -1
            row = e * res_tok + p % res_tok
            return row if B + 1 + row <= INT32_MAX else None

        # Validation (readings R6 and R14).
        err = 0
        seen = set()
        for p in sel:
            if p == -1:
                continue
            if p < -1 or p >= P:
                err |= ERR_RANGE
                continue
            rr = resident_row(p)
            if rr is None:
                err |= ERR_RANGE
                continue
            if rr >= 0:
                continue                   # never reaches the hot tier (R14)
            if p in seen and not union:
                err |= ERR_DUP
            seen.add(p)
        if newest < -1 or newest >= P:
            err |= ERR_RANGE
        if err:
            self.miss_count = 0            # nothing was fetched this step
            return [-1] * k, [], err

        # Stages 1-2: classify every selection as padding, resident, newest,
        # hit or miss.
        out = [None] * k
        hit_slots = set()
        misses = []                        # selection indices, in list order
        first = {}                         # union mode: position -> first index
        for i, p in enumerate(sel):
            if union and p != -1 and p in first:
                continue                   # a later reference: filled in below
            first[p] = i
            if p == -1:
                out[i] = -1
            elif resident_row(p) >= 0:
                out[i] = B + 1 + resident_row(p)   # reading R14
            elif newest >= 0 and p == newest:
                out[i] = B                 # reading R4
            elif p in self.page_table:
                s = self.page_table[p]
                out[i] = s
                hit_slots.add(s)
            else:
                misses.append(i)

        # Stage 3: evictable slots in LRU order; miss j takes the j-th oldest.
        ev = [s for s in self.lru if s not in hit_slots]
        M = len(misses)
        assert M <= len(ev), "B >= k guarantees a victim for every miss"

        # Stages 4-5: fetch into the victims and publish the new mapping.
        plan = []
        for j, i in enumerate(misses):
            s = ev[j]
            p = sel[i]
            old = self.slot_pos[s]
            if old >= 0:
                del self.page_table[old]
            self.slot_pos[s] = p
            self.page_table[p] = s
            if self.host is not None and not skip_io:
                self.hot[s] = self.host(p)
            out[i] = s
            plan.append((p, s))

        if union:                          # later references share the first's row
            for i, p in enumerate(sel):
                if out[i] is None:
                    out[i] = out[first[p]]

        # New recency order: untouched evictables (oldest), then this step's
        # fetches, then this step's hits (newest) -- [P1] §3.3 and the worked
        # example of [P1] §3.5; readings R1 and R2 fix the order inside groups.
        self.lru = ev[M:] + ev[:M] + sorted(hit_slots)
        self.miss_count = M
        return out, plan, 0

    # ------------------------------------------------------------------ #
    def resolve_short(self, sel, newest, seq_len, prev=-1, res_blocks=None, res_tok=1):
        """Short-request step (reading R17; caller checks seq_len <= B): grow
        by ``prev`` (when >= 0; the host must already hold its record), then
        look the selections up by position.  Returns ``(out, plan, err)``;
        ``plan`` is the growth's."""
        B, P = self.B, self.P
        plan = []
        if prev >= 0:
            _, plan, e = self.resolve([prev])
            assert e == 0, "the previous token must be a position in [0, P)"
        else:
            self.miss_count = 0
        err = 0
        if newest < -1 or newest >= P:
            err |= ERR_RANGE
        out = []
        for p in sel:
            if p == -1:
                out.append(-1)
                continue
            if p < -1 or p >= P:
                err |= ERR_RANGE
                out.append(-1)
                continue
            row = -1
            if res_blocks is not None and p // res_tok < len(res_blocks):
                e = res_blocks[p // res_tok]
                if e < -1:
                    err |= ERR_RANGE
                    out.append(-1)
                    continue
                if e >= 0:
                    row = e * res_tok + p % res_tok
                    if B + 1 + row > INT32_MAX:
                        err |= ERR_RANGE
                        out.append(-1)
                        continue
            if row >= 0:
                out.append(B + 1 + row)
            elif newest >= 0 and p == newest:
                out.append(B)
            elif p >= seq_len:
                err |= ERR_RANGE
                out.append(-1)
            else:
                out.append(p)                  # slot numbered like the position
        if err:
            out = [-1] * len(sel)
        return out, plan, err

    # ------------------------------------------------------------------ #
    def admit(self, n, k=None):
        """Admission of a request (gentlecold.top §5.3, direct admission:
        a long request starts with every token marked absent -- the reset
        state, n = 0 -- and a short one, host length <= the buffer, is
        preloaded).  Reading R16: preloading the first ``n`` positions gives
        the state that resolving positions 0, 1, ..., n-1 in order from the
        reset state gives, whether in one list or in consecutive lists of
        ``k``: slot s holds position s, and the LRU order is the empty slots
        (ascending) followed by the preloaded ones (ascending)."""
        B = self.B
        if not 0 <= n <= min(B, self.P):
            raise ValueError("preload length outside [0, min(B, P)]")
        self.slot_pos = [-1] * B
        self.lru = list(range(B))
        self.page_table = {}
        self.hot = [None] * (B + 1)
        self.miss_count = 0
        k = k or max(1, n)
        plan = []
        for c0 in range(0, n, k):
            chunk = list(range(c0, min(n, c0 + k)))
            out, pl, err = self.resolve(chunk + [-1] * (k - len(chunk)))
            assert err == 0
            plan += pl
        self.miss_count = 0                # an admission is not a decode step
        return plan


def expand_blocks(sel_blocks, block_tokens):
    """Token positions of a block-id selection list (gentlecold.top §5.5: a
    selector that picks blocks; the kernel expands each block id into its
    positions).  Block b stands for positions b*block_tokens .. b*block_tokens
    + block_tokens - 1, in that order; -1 stands for block_tokens paddings.
    Any other negative id gives negative positions, which the resolve rejects
    as out of range."""
    out = []
    for b in sel_blocks:
        if b == -1:
            out.extend([-1] * block_tokens)
        else:
            out.extend(b * block_tokens + j for j in range(block_tokens))
    return out


# ---------------------------------------------------------------------- #
# Brute-force optimal replacement (Belady's offline optimum), for bounds.  #
# ---------------------------------------------------------------------- #
def optimal_misses(trace, B):
    """Fewest misses any replacement policy with ``B`` slots can reach.

    Exhaustive search over which resident positions to keep at each step.
    The positions selected in the current step must all be resident after
    it (they are protected), and a miss is a selected position that was not
    resident before the step.  Only for tiny traces (B <= 4, a handful of
    positions and steps).
    """
    from functools import lru_cache
    from itertools import combinations

    steps = [frozenset(p for p in s if p != -1) for s in trace]

    @lru_cache(maxsize=None)
    def best(t, resident):
        if t == len(steps):
            return 0
        S = steps[t]
        if len(S) > B:
            raise ValueError("selection larger than B")
        cost = len(S - resident)
        others = sorted(resident - S)
        room = B - len(S)
        keep_n = min(room, len(others))
        # Keeping more never hurts, so only maximal keep-sets are searched.
        return cost + min(best(t + 1, S | frozenset(keep))
                          for keep in combinations(others, keep_n))

    return best(0, frozenset())
