"""CUDA path == oracle, bit for bit, through the C ABI (needs a GB300)."""
import itertools

import numpy as np
import pytest
import torch

from host_offload_serving_gb300 import hisparse as H
from host_offload_serving_gb300.runtime import HiSparse, WorkloadMemory
from oracle.coracle import OracleLayer
from workload import get, sweep_workload
import pins

pytestmark = pytest.mark.gpu


LOOKUPS = [H.LOOKUP_PAGE_TABLE, H.LOOKUP_HASH]


def _instance(R, k, B, P, rec=16, ctas=0, fill=None, lookup=H.LOOKUP_PAGE_TABLE):
    mem = WorkloadMemory(R, 1, B, P, rec)
    host = mem.host_view(0)
    if fill is None:
        host[:] = np.random.default_rng(R * 1000 + k).integers(0, 256, size=host.shape, dtype=np.uint8)
    hs = HiSparse(R, 1, k, B, P, rec, mem.layer_buffers(), ctas_per_request=ctas, lookup=lookup)
    return mem, hs


def _dev(a, dtype=torch.int32):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda").to(dtype)


# ---------------------------------------------------------------------- #
@pytest.mark.parametrize("lookup", LOOKUPS)
def test_worked_example_b(lookup):
    """gentlecold.top deep dive §3.5 worked example, preset through import."""
    g = dict(pins.parse_golden("example_b_resolve.txt"))
    B, k, P = int(g["B"]), int(g["k"]), 64
    mem, hs = _instance(1, k, B, P, lookup=lookup)
    sp = np.array([pins._ints(g["slot_pos"])], np.int32)
    lru = np.array([pins._ints(g["lru"])], np.int16)
    pt = np.full((1, P), -1, np.int32)
    for s, p in enumerate(sp[0]):
        pt[0, p] = s
    assert hs.import_state(0, sp, lru, pt) == 0
    sel = _dev(np.array([pins._ints(g["sel"])], np.int32))
    newest = _dev(np.array([int(g["newest"])], np.int32))
    out = torch.empty((1, k), dtype=torch.int32, device="cuda")
    hs.resolve(0, sel, out, newest=newest, flags=H.RECORD_PLAN)
    torch.cuda.synchronize()
    assert out.cpu().numpy()[0].tolist() == pins._ints(g["expect_out"])
    sp2, lru2, pt2, mc = hs.export_state(0)
    assert lru2[0].tolist() == pins._ints(g["expect_lru"])
    assert sp2[0].tolist() == pins._ints(g["expect_slot_pos"])
    assert mc[0] == int(g["expect_misses"])
    c, pp, ps = hs.export_plan(0)
    assert c[0] == 1 and (pp[0, 0], ps[0, 0]) == (25, 0)
    assert pt2[0, 25] == 0 and pt2[0, 10] == -1 and pt2[0, 12] == 2
    host = mem.host_view(0)
    assert (mem.hot[0, 0, 0].cpu().numpy() == host[0, 25]).all()
    hs.close(); mem.close()


@pytest.mark.parametrize("lookup", LOOKUPS)
def test_worked_example_a(lookup):
    """notes.kuangjux.top §5: misses 3,1,1 at capacity 3 and 3,1,0 at capacity 4."""
    rows = pins.parse_golden("example_a_capacity.txt")
    steps = [pins._ints(v) for key, v in rows if key == "step"]
    for cap, exp in ((3, [3, 1, 1]), (4, [3, 1, 0])):
        mem, hs = _instance(1, 3, cap, 16, lookup=lookup)
        out = torch.empty((1, 3), dtype=torch.int32, device="cuda")
        got = []
        for s in steps:
            hs.resolve(0, _dev(np.array([s], np.int32)), out)
            got.append(int(hs.export_state(0)[3][0]))
        assert got == exp
        hs.close(); mem.close()


# ---------------------------------------------------------------------- #
def _enumerate_lists(k, P):
    """Every selection list of length k over positions [0, P) with -1 padding."""
    out = []
    for m in range(k + 1):
        for vals in itertools.permutations(range(P), m):
            for slots in itertools.combinations(range(k), m):
                row = [-1] * k
                for s, v in zip(slots, vals):
                    row[s] = v
                out.append(row)
    return out


@pytest.mark.parametrize("lookup", LOOKUPS)
@pytest.mark.parametrize("k,P,steps,extra", [(2, 4, 3, (0, 1, 2)), (3, 5, 2, (0, 1)),
                                              (1, 4, 4, (0, 1, 2))])
def test_exhaustive_tiny(k, P, steps, extra, lookup):
    """All selection sequences of a tiny domain, one sequence per request."""
    lists = _enumerate_lists(k, P)
    seqs = list(itertools.product(range(len(lists)), repeat=steps))
    for B in (k + e for e in extra):
        for start in range(0, len(seqs), 8192):
            chunk = seqs[start:start + 8192]
            R = len(chunk)
            sel = np.array([[lists[i] for i in s] for s in chunk], np.int32)  # [R][T][k]
            sel = np.ascontiguousarray(sel.transpose(1, 0, 2))               # [T][R][k]
            newest = np.where(np.arange(R) % 3 == 0, P - 1, -1).astype(np.int32)
            mem, hs = _instance(R, k, B, P, lookup=lookup, ctas=1 + (R % 3 == 1))
            host = mem.host_view(0)
            o = OracleLayer(R, k, B, P, 16, host=host)
            o.reset()
            out = torch.empty((R, k), dtype=torch.int32, device="cuda")
            dnew = _dev(newest)
            for t in range(steps):
                hs.resolve(0, _dev(sel[t]), out, newest=dnew)
                oo, e = o.resolve(sel[t], newest)
                assert e == 0
                np.testing.assert_array_equal(out.cpu().numpy(), oo)
            sp, lru, pt, mc = hs.export_state(0)
            np.testing.assert_array_equal(sp, o.slot_pos)
            np.testing.assert_array_equal(lru, o.lru)
            np.testing.assert_array_equal(pt, o.page_table)
            np.testing.assert_array_equal(mc, o.miss_count)
            np.testing.assert_array_equal(mem.hot[0].cpu().numpy()[:, :B], o.hot[:, :B])
            hs.close(); mem.close()


# ---------------------------------------------------------------------- #
from harness import Run  # noqa: E402


def _run_all(w, every=1, **kw):
    """Run every step on both sides.  Slot vectors and miss counts are
    compared after every step; the full state (slot map, LRU, page table,
    plan, every hot byte, written-back rows) after every ``every``-th step and
    the last; the untouched prefill host rows at the first full compare and
    the last."""
    run = Run(w, **kw)
    try:
        for t in range(w.steps):
            run.step()
            if t % every == 0 or t == w.steps - 1:
                run.compare(check_prefill=(t == 0 or t == w.steps - 1))
            else:
                run.compare_light()
    finally:
        run.close()


def test_tiny_workload_every_step():
    _run_all(get("tiny"))


@pytest.mark.parametrize("lookup", LOOKUPS)
def test_dsa_workload_full_size_every_step(lookup):
    """8 requests x 4 layers, 128K context, k=2048, B=4096, write-through
    fused into RESOLVE."""
    _run_all(get("dsa"), lookup=lookup)


@pytest.mark.parametrize("lookup", LOOKUPS)
def test_separate_writeback_launch(lookup):
    """The write-through as its own launch on a backup stream (the pages' order)."""
    _run_all(get("dsa").scaled(R=4, groups=2, L_ctx=32768, steps=8), lookup=lookup, fused=False)


@pytest.mark.parametrize("mode", ["group", "layer", "inline"])
def test_write_through_with_shared_layers(mode):
    """Write-through on anchors (fused) and on shared layers (own launch)."""
    _run_all(get("shared").scaled(R=3, groups=2, L_ctx=8192, steps=6, write_through=True),
             group_replay=mode == "group", inline_shared=mode == "inline")


def test_quest_workload_scaled():
    """Page granularity with 32 KB records (fewer requests/layers/pages)."""
    _run_all(get("quest").scaled(R=4, groups=2, L_ctx=2048, steps=12))


@pytest.mark.parametrize("mode", ["group", "layer", "inline"])
def test_shared_workload_scaled(mode):
    """Anchor + 3 shared layers (fewer requests, shorter context): one replay
    launch per group, one per shared layer, or the shared layers filled
    inside the anchor's RESOLVE."""
    _run_all(get("shared").scaled(R=6, groups=2, L_ctx=16384, steps=10),
             group_replay=mode == "group", inline_shared=mode == "inline")


@pytest.mark.parametrize("followers", [1, 8, 11])
def test_group_replay_many_layers(followers):
    """One anchor with 1, 8 (one launch) and 11 (two launches) shared layers."""
    _run_all(get("shared").scaled(R=3, groups=1, followers=followers, L_ctx=4096, steps=5),
             replay_ctas=3)


@pytest.mark.parametrize("cs", [1, 3, 0])
@pytest.mark.parametrize("followers", [1, 8])
def test_inline_shared_layers(followers, cs):
    """Shared layers filled inside the anchor's launch, every cluster shape."""
    _run_all(get("shared").scaled(R=3, groups=2, followers=followers, L_ctx=4096, steps=5),
             inline_shared=True, ctas_per_request=cs)


def test_inline_shared_from_mirror_and_limits():
    """FROM_MIRROR reads every layer's mirror; 9 shared layers are refused
    (EBOUND); the hash lookup refuses the flag (EINVAL)."""
    _run_all(get("shared").scaled(R=2, groups=1, L_ctx=2048, steps=4), inline_shared=True,
             flags=H.FROM_MIRROR, mirror=True)
    for followers, lookup, code in ((9, H.LOOKUP_PAGE_TABLE, H.EBOUND),
                                    (2, H.LOOKUP_HASH, H.EINVAL)):
        w = get("shared").scaled(R=2, groups=1, followers=followers, L_ctx=1024, steps=2)
        mem = WorkloadMemory(w.R, w.L, w.B, w.P, w.rec)
        hs = HiSparse(w.R, w.L, w.k, w.B, w.P, w.rec, mem.layer_buffers(),
                      anchor_of=w.anchor_of(), lookup=lookup)
        sel = torch.full((w.R, w.k), -1, dtype=torch.int32, device="cuda")
        out = torch.empty((w.R, w.k), dtype=torch.int32, device="cuda")
        with pytest.raises(H.HiSparseError) as ei:
            hs.resolve(0, sel, out, flags=H.WITH_SHARED)
        assert ei.value.code == code
        torch.cuda.synchronize()
        hs.close(); mem.close()


def test_group_replay_roles():
    """follower -1 on an anchor without shared layers launches nothing; a
    shared layer as the anchor, or another anchor's layer, is refused."""
    w = get("shared").scaled(R=2, groups=2, L_ctx=1024, steps=2)
    mem = WorkloadMemory(w.R, w.L, w.B, w.P, w.rec)
    hs = HiSparse(w.R, w.L, w.k, w.B, w.P, w.rec, mem.layer_buffers(), anchor_of=w.anchor_of())
    assert H.hisparse_prefetch_plan(hs.h, 1, -1, None, None) == H.EROLE
    assert H.hisparse_prefetch_plan(hs.h, 0, 5, None, None) == H.EROLE
    assert H.hisparse_prefetch_plan(hs.h, 0, -2, None, None) == H.EINVAL
    assert H.hisparse_prefetch_plan(hs.h, w.L, -1, None, None) == H.EINVAL
    hs.close(); mem.close()
    w = get("dsa").scaled(R=2, groups=2, L_ctx=1024, steps=2)
    mem = WorkloadMemory(w.R, w.L, w.B, w.P, w.rec)
    hs = HiSparse(w.R, w.L, w.k, w.B, w.P, w.rec, mem.layer_buffers(), anchor_of=w.anchor_of())
    assert H.hisparse_prefetch_plan(hs.h, 0, -1, None, None) == H.OK
    torch.cuda.synchronize()
    hs.close(); mem.close()


@pytest.mark.parametrize("B", [2048, 4096, 8192])
def test_sweep_workload_scaled(B):
    _run_all(sweep_workload(B, 0.70, L_ctx=65536).scaled(R=4, steps=6))


@pytest.mark.parametrize("lookup", LOOKUPS)
@pytest.mark.parametrize("cs", [1, 2, 3, 4, 8, 16])
def test_cluster_sizes_identical(cs, lookup):
    _run_all(get("dsa").scaled(R=3, groups=1, L_ctx=16384, steps=5), ctas_per_request=cs,
             lookup=lookup)


@pytest.mark.parametrize("lookup", LOOKUPS)
def test_skip_io_metadata_identical_bytes_stale(lookup):
    _run_all(get("dsa").scaled(R=2, groups=2, L_ctx=8192, steps=5), flags=H.SKIP_IO, lookup=lookup)


def test_from_mirror_bytes_identical():
    _run_all(get("quest").scaled(R=2, groups=1, L_ctx=1024, steps=5), flags=H.FROM_MIRROR,
             mirror=True)


@pytest.mark.parametrize("lookup", LOOKUPS)
@pytest.mark.parametrize("fused", [True, False])
def test_from_mirror_with_write_through(lookup, fused):
    """FROM_MIRROR with the write-through on (DSA-style: the previous token
    sits in the local window, so it is selected again right after its
    write-back): every write-back also lands in the HBM mirror, so the
    mirror-fed fetches return the written bytes.  Every step is compared with
    the oracle, and at the end the mirror equals the host pool byte for byte."""
    w = get("dsa").scaled(R=3, groups=2, L_ctx=8192, steps=8)
    run = Run(w, lookup=lookup, fused=fused, mirror=True, flags=H.FROM_MIRROR)
    try:
        for t in range(w.steps):
            run.step()
            run.compare(check_prefill=(t == w.steps - 1))
        pool = run.mem.pool.numpy()[:run.mem.mirror.numel()]
        assert np.array_equal(run.mem.mirror.cpu().numpy(), pool), "mirror differs from pool"
    finally:
        run.close()


@pytest.mark.parametrize("mode", ["group", "inline"])
def test_from_mirror_with_write_through_shared_layers(mode):
    """The same on shared-index layers, whose write-backs are their own
    launches (and the anchors' fused)."""
    _run_all(get("shared").scaled(R=2, groups=2, L_ctx=4096, steps=6, write_through=True),
             mirror=True, flags=H.FROM_MIRROR, inline_shared=mode == "inline",
             group_replay=mode == "group")


def test_l2_persisting_page_tables_change_nothing():
    """With the page tables kept persisting in L2, every step equals the
    oracle; turning it off again works; a negative size is refused."""
    w = get("dsa").scaled(R=3, groups=2, L_ctx=16384, steps=6)
    _run_all(w, l2_persist=16 << 20)
    mem = WorkloadMemory(w.R, w.L, w.B, w.P, w.rec)
    hs = HiSparse(w.R, w.L, w.k, w.B, w.P, w.rec, mem.layer_buffers())
    assert H.hisparse_set_l2_persisting(hs.h, -1) == H.EINVAL
    assert H.hisparse_set_l2_persisting(hs.h, 8 << 20) == H.OK
    assert H.hisparse_set_l2_persisting(hs.h, 0) == H.OK
    hs.close(); mem.close()


def test_huge_page_pool():
    """The same results from a huge-page-backed, registered host pool."""
    _run_all(get("dsa").scaled(R=3, groups=2, L_ctx=65536, steps=6), pool_kind=H.HOST_HUGE)


def test_num_reqs_padding_leaves_tail_untouched():
    _run_all(get("dsa").scaled(R=5, groups=1, L_ctx=8192, steps=4), num_reqs=3)


# ---------------------------------------------------------------------- #
@pytest.mark.parametrize("lookup", LOOKUPS)
@pytest.mark.parametrize("cs", [1, 3])
def test_device_detected_errors_keep_state(lookup, cs):
    R, k, B, P = 4, 4, 6, 32
    mem, hs = _instance(R, k, B, P, lookup=lookup, ctas=cs)
    out = torch.empty((R, k), dtype=torch.int32, device="cuda")
    good = np.array([[1, 2, 3, -1]] * R, np.int32)
    hs.resolve(0, _dev(good), out)
    before = hs.export_state(0)
    bad = np.array([[4, 4, 5, -1],      # duplicate
                    [4, 32, 5, -1],     # out of range
                    [4, -9, 5, -1],     # out of range
                    [7, 8, 9, 10]], np.int32)
    hs.resolve(0, _dev(bad), out)
    o = out.cpu().numpy()
    assert (o[:3] == -1).all() and (o[3] >= 0).all()
    flags, ue = hs.status()
    assert flags == (H.ERR_DUP | H.ERR_RANGE)
    assert ue[0].tolist() == [H.ERR_DUP, H.ERR_RANGE, H.ERR_RANGE, 0]
    after = hs.export_state(0)
    for r in range(3):
        for a, b in zip(before[:3], after[:3]):      # slot_pos, lru, page table
            np.testing.assert_array_equal(a[r], b[r])
    assert after[3][:3].tolist() == [0, 0, 0]        # nothing fetched for failed units
    assert hs.status()[0] == 0     # reading clears the word
    newest = _dev(np.array([40, -1, -1, -1], np.int32))
    hs.resolve(0, _dev(good), out, newest=newest)
    assert hs.status()[0] == H.ERR_RANGE
    hs.close(); mem.close()


@pytest.mark.parametrize("cs", [1, 2])
@pytest.mark.parametrize("m", [20, 100, 500])
def test_duplicate_among_one_slices_misses(cs, m):
    """A repeated position whose two copies are both misses of the same slice
    fails the unit with its admission state untouched, whichever way the slice
    orders its fetch list (one warp, direct ranks, row buckets); the same list
    without the repeat then resolves exactly as the oracle does."""
    R, k, B, P, rec = 1, 512, 1024, 8192, 16
    mem, hs = _instance(R, k, B, P, rec=rec, ctas=cs)
    out = torch.empty((R, k), dtype=torch.int32, device="cuda")
    pos = np.random.default_rng(m).choice(P, size=m, replace=False).astype(np.int32)
    bad = np.full((R, k), -1, np.int32)
    bad[0, :m] = pos
    bad[0, m - 1] = pos[0]
    hs.resolve(0, _dev(bad), out)
    flags, ue = hs.status()
    assert flags == H.ERR_DUP and ue[0].tolist() == [H.ERR_DUP]
    assert (out.cpu().numpy() == -1).all()
    sp, lru, pt, mc = hs.export_state(0)
    assert (sp == -1).all() and (pt == -1).all() and mc.tolist() == [0]
    assert lru[0].tolist() == list(range(B))
    good = bad.copy()
    good[0, m - 1] = -1
    hs.resolve(0, _dev(good), out)
    ora = OracleLayer(R, k, B, P, rec, host=mem.host_view(0))
    o_out, o_err = ora.resolve(good)
    assert hs.status()[0] == 0 and not np.any(o_err)
    np.testing.assert_array_equal(out.cpu().numpy(), o_out)
    sp, lru, pt, mc = hs.export_state(0)
    np.testing.assert_array_equal(sp, ora.slot_pos)
    np.testing.assert_array_equal(lru, ora.lru)
    np.testing.assert_array_equal(pt, ora.page_table)
    np.testing.assert_array_equal(mc, ora.miss_count)
    np.testing.assert_array_equal(mem.hot[0].cpu().numpy()[:, :B], ora.hot[:, :B])
    hs.close(); mem.close()


# ---------------------------------------------------------------------- #
# Three-tier resolve: resident block table first                          #
# ---------------------------------------------------------------------- #
from workload.resident import resident_tables  # noqa: E402


@pytest.mark.parametrize("cs", [0, 1, 3])
def test_resident_tier_small(cs):
    """One request wholly resident, the others with a resident recent window,
    write-through fused; state, slot vectors and bytes equal the oracle's."""
    w = get("dsa").scaled(R=4, groups=2, L_ctx=16384, steps=8)
    _run_all(w, ctas_per_request=cs, resident=(resident_tables(w, 64, full=1, window=1024), 64))


def test_resident_tier_dsa_full_size():
    """The DSA-style workload at full size with half the requests resident."""
    w = get("dsa")
    _run_all(w, every=4, resident=(resident_tables(w, 64, full=4, window=4096), 64))


@pytest.mark.parametrize("inline", [False, True])
def test_resident_tier_shared_layers(inline):
    """Anchors resolved with the resident tier; shared layers replay their
    plans, or are filled inside the anchor's launch."""
    w = get("shared").scaled(R=3, groups=2, L_ctx=8192, steps=6)
    _run_all(w, resident=(resident_tables(w, 16, full=1, window=512), 16), inline_shared=inline)


def test_resident_all_and_errors():
    """A wholly resident request keeps its state; a bad block entry fails only
    the request that selects a position in it; repeats of a resident position
    are not duplicates."""
    R, k, B, P, tok = 3, 8, 16, 256, 16
    mem, hs = _instance(R, k, B, P)
    out = torch.empty((R, k), dtype=torch.int32, device="cuda")
    warm = np.array([[1, 2, 3, 4, 5, 6, 7, 8]] * R, np.int32)
    hs.resolve(0, _dev(warm), out)
    before = hs.export_state(0)
    blocks = np.full((R, P // tok), -1, np.int32)
    blocks[0, :] = np.arange(P // tok) + 100          # request 0: everything resident
    blocks[1, 2] = -5                                  # request 1: a bad entry in block 2
    blocks[2, 0] = 7                                   # request 2: block 0 resident
    sel = np.array([[1, 40, 41, 200, 7, -1, 90, 3],
                    [1, 33, 2, -1, -1, -1, -1, -1],    # 33 is in block 2
                    [1, 1 + 0, 40, 50, -1, -1, -1, -1]], np.int32)
    sel[2, 1] = 1                                      # a repeat of a resident position
    hs.resolve_resident(0, _dev(sel), out, _dev(blocks), tok)
    o = out.cpu().numpy()
    assert o[0].tolist() == [B + 1 + 100 * tok + 1, B + 1 + 102 * tok + 8, B + 1 + 102 * tok + 9,
                             B + 1 + 112 * tok + 8, B + 1 + 100 * tok + 7, -1,
                             B + 1 + 105 * tok + 10, B + 1 + 100 * tok + 3]
    assert (o[1] == -1).all()
    assert o[2, 0] == o[2, 1] == B + 1 + 7 * tok + 1
    flags, ue = hs.status()
    assert flags == H.ERR_RANGE and ue[0].tolist() == [0, H.ERR_RANGE, 0]
    after = hs.export_state(0)
    for r in (0, 1):
        for x, y in zip(before[:3], after[:3]):
            np.testing.assert_array_equal(x[r], y[r])
    assert after[3][2] == 2                            # request 2 fetched 40 and 50
    hs.close(); mem.close()


# ---------------------------------------------------------------------- #
# Block-id selections expanded in the kernel                               #
# ---------------------------------------------------------------------- #
@pytest.mark.parametrize("cs", [0, 1, 5])
def test_block_selections_small(cs):
    """Top-k blocks of 4 positions, read as block ids by the kernel; the
    oracle resolves the expanded positions."""
    _run_all(get("blocks").scaled(R=3, groups=2, L_ctx=16384, steps=8), ctas_per_request=cs)


def test_block_selections_full_size():
    """8 requests x 4 layers, 128K context, top-512 blocks of 4 positions."""
    _run_all(get("blocks"), every=4)


def test_block_selections_with_resident_tier():
    w = get("blocks").scaled(R=3, groups=2, L_ctx=8192, steps=6)
    _run_all(w, resident=(resident_tables(w, 16, full=1, window=256), 16))


def test_block_selection_errors():
    """A negative block id other than -1 and a block past P fail the request;
    -1 blocks are padding."""
    R, k, B, P, bt = 3, 8, 16, 64, 4
    mem, hs = _instance(R, k, B, P)
    out = torch.empty((R, k), dtype=torch.int32, device="cuda")
    blocks = np.array([[2, -1], [3, -2], [15, 16]], np.int32)   # 16 * 4 = 64 = P
    hs.resolve_ex(0, _dev(blocks), out, sel_block_tokens=bt)
    o = out.cpu().numpy()
    sp = hs.export_state(0)[0]
    assert o[0, :4].tolist() == sorted(o[0, :4].tolist()) and (o[0, 4:] == -1).all()
    assert [int(sp[0, s]) for s in o[0, :4]] == [8, 9, 10, 11]
    assert (o[1] == -1).all() and (o[2] == -1).all()
    flags, ue = hs.status()
    assert flags == H.ERR_RANGE and ue[0].tolist() == [0, H.ERR_RANGE, H.ERR_RANGE]
    hs.close(); mem.close()


# ---------------------------------------------------------------------- #
# Union mode: speculative verify rows resolved together                   #
# ---------------------------------------------------------------------- #
def _verify_row_traces(w, V):
    from workload.traces import verify_row_traces
    return verify_row_traces(w, V)


@pytest.mark.parametrize("cs", [0, 1, 3])
def test_union_verify_rows_small(cs):
    w = get("dsa").scaled(R=3, groups=2, L_ctx=16384, steps=8, k=512, B=1024,
                          write_through=False)
    _run_all(w, traces=_verify_row_traces(w, 4), flags=H.UNION, ctas_per_request=cs)


def test_union_verify_rows_full_size():
    """8 requests x 4 layers, 4 verify rows of 512 selections (2048 in all), B=4096."""
    w = get("dsa").scaled(write_through=False)
    _run_all(w, every=4, traces=_verify_row_traces(w, 4), flags=H.UNION)


@pytest.mark.parametrize("inline", [False, True])
def test_union_with_shared_layers_and_resident_tier(inline):
    """Repeated misses (union) are fetched once for the shared layers too."""
    w = get("shared").scaled(R=3, groups=2, L_ctx=8192, steps=6, k=512, B=1024)
    _run_all(w, traces=_verify_row_traces(w, 2), flags=H.UNION,
             resident=(resident_tables(w, 16, full=0, window=256), 16), inline_shared=inline)


def test_union_repeats_are_not_errors():
    R, k, B, P = 2, 8, 16, 64
    mem, hs = _instance(R, k, B, P)
    out = torch.empty((R, k), dtype=torch.int32, device="cuda")
    sel = np.array([[1, 2, 3, 3, 4, 1, -1, 2],
                    [5, 5, 5, 5, 70, -1, -1, -1]], np.int32)     # 70 >= P: still an error
    hs.resolve(0, _dev(sel), out, flags=H.UNION)
    o = out.cpu().numpy()
    assert o[0].tolist() == [0, 1, 2, 2, 3, 0, -1, 1]
    assert (o[1] == -1).all()
    flags, ue = hs.status()
    assert flags == H.ERR_RANGE and ue[0].tolist() == [0, H.ERR_RANGE]
    assert hs.export_state(0)[3].tolist() == [4, 0]
    hs.close(); mem.close()


# ---------------------------------------------------------------------- #
# Admission with preload                                                   #
# ---------------------------------------------------------------------- #
@pytest.mark.parametrize("name", ["shared", "dsa"])
def test_admit_between_steps(name):
    """Requests admitted mid-run (one preloaded, one direct with nothing
    preloaded, one preloaded to the full buffer) then decoded: every field
    equals the oracle's after the admission and after each later step."""
    w = get(name).scaled(R=4, groups=2, L_ctx=8192, steps=8, k=256, B=512)
    run = Run(w)
    try:
        for t in range(3):
            run.step()
        run.admit([1, 3, 0], [300, 0, 512])
        run.compare()
        for t in range(3, w.steps):
            run.step()
            run.compare()
    finally:
        run.close()


def test_admit_rejects_bad_entries():
    R, k, B, P = 3, 4, 8, 64
    mem, hs = _instance(R, k, B, P)
    out = torch.empty((R, k), dtype=torch.int32, device="cuda")
    hs.resolve(0, _dev(np.array([[1, 2, 3, 4]] * R, np.int32)), out)
    before = hs.export_state(0)
    hs.admit(0, _dev(np.array([5, 1], np.int32)), _dev(np.array([2, 9], np.int32)))
    flags, _ = hs.status()
    assert flags == H.ERR_RANGE                      # request 5 >= R, preload 9 > B
    after = hs.export_state(0)
    for x, y in zip(before[:3], after[:3]):
        np.testing.assert_array_equal(x, y)
    hs.admit(0, _dev(np.array([2], np.int32)), _dev(np.array([3], np.int32)))
    sp, lru, pt, mc = hs.export_state(0)
    assert sp[2].tolist() == [0, 1, 2, -1, -1, -1, -1, -1]
    assert lru[2].tolist() == [3, 4, 5, 6, 7, 0, 1, 2] and mc[2] == 0
    assert pt[2, :4].tolist() == [0, 1, 2, -1] and (pt[2, 4:] == -1).all()
    host = mem.host_view(0)
    np.testing.assert_array_equal(mem.hot[0, 2, :3].cpu().numpy(), host[2, :3])
    hs.close(); mem.close()


# ---------------------------------------------------------------------- #
# Host pools with a shared-index group's layers interleaved row by row    #
# ---------------------------------------------------------------------- #
@pytest.mark.parametrize("mode", ["group", "layer", "inline"])
def test_group_interleaved_host_layout_shared(mode):
    """Anchor + 3 shared layers with their host rows interleaved: same results."""
    _run_all(get("shared").scaled(R=4, groups=2, L_ctx=16384, steps=8), group=4,
             group_replay=mode == "group", inline_shared=mode == "inline")


def test_group_interleaved_host_layout_write_through():
    """Interleaved rows with the fused write-through and shared-layer write-backs."""
    _run_all(get("shared").scaled(R=3, groups=2, L_ctx=8192, steps=6, write_through=True),
             group=4)


def test_hash_lookup_rejects_extended_options():
    """The hash-lookup kernel has no resident tier, block ids or union mode."""
    R, k, B, P = 2, 8, 16, 64
    mem, hs = _instance(R, k, B, P, lookup=H.LOOKUP_HASH)
    out = torch.empty((R, k), dtype=torch.int32, device="cuda")
    sel = _dev(np.array([[1, 2, 3, 4, 5, 6, 7, 8]] * R, np.int32))
    blocks = _dev(np.full((R, 4), -1, np.int32))
    with pytest.raises(H.HiSparseError):
        hs.resolve_ex(0, sel, out, res_blocks=blocks, res_block_tokens=16)
    with pytest.raises(H.HiSparseError):
        hs.resolve_ex(0, _dev(np.array([[1, 2]] * R, np.int32)), out, sel_block_tokens=4)
    with pytest.raises(H.HiSparseError):
        hs.resolve(0, sel, out, flags=H.UNION)
    hs.resolve(0, sel, out)                       # the plain call still works
    assert hs.status()[0] == 0
    hs.close(); mem.close()


def test_import_rejects_inconsistent_state():
    mem, hs = _instance(1, 2, 4, 16)
    sp = np.array([[3, -1, 5, -1]], np.int32)
    lru = np.array([[0, 1, 2, 3]], np.int16)
    pt = np.full((1, 16), -1, np.int32)
    pt[0, 3], pt[0, 5] = 0, 2
    assert hs.import_state(0, sp, lru, pt) == 0
    pt[0, 5] = 1
    assert hs.import_state(0, sp, lru, pt) == H.EINVAL
    pt[0, 5] = 2
    assert hs.import_state(0, sp, np.array([[0, 1, 1, 3]], np.int16), pt) == H.EINVAL
    # miss counts: imported with the rest, validated against [0, k]
    assert hs.import_state(0, sp, lru, pt, np.array([3], np.int32)) == H.EINVAL
    assert hs.export_state(0)[3].tolist() == [0]
    assert hs.import_state(0, sp, lru, pt, np.array([2], np.int32)) == 0
    sp2, lru2, pt2, mc2 = hs.export_state(0)
    assert sp2.tolist() == sp.tolist() and lru2.tolist() == lru.tolist()
    assert pt2.tolist() == pt.tolist() and mc2.tolist() == [2]
    hs.close(); mem.close()


def test_export_import_round_trip_mid_run():
    """Checkpoint / resume: a run's state exported after some steps and
    imported into a fresh instance (with the hot bytes copied) continues
    exactly as the uninterrupted run does."""
    w = get("dsa").scaled(R=3, groups=1, L_ctx=8192, steps=8, write_through=False)
    a = Run(w)
    b = Run(w)
    try:
        for t in range(4):
            a.step()
        for l, _ in a.groups:
            assert b.hs.import_state(l, *a.hs.export_state(l)) == 0
        b.mem.hot.copy_(a.mem.hot)
        for l, _ in a.groups:
            np.testing.assert_array_equal(b.hs.export_state(l)[3], a.hs.export_state(l)[3])
        for t in range(4, w.steps):
            a.step()
            b.gpu_step(t)
        a.compare()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(b.out.cpu().numpy(), a.out.cpu().numpy())
        for l, _ in a.groups:
            for x, y in zip(a.hs.export_state(l), b.hs.export_state(l)):
                np.testing.assert_array_equal(x, y)
        assert torch.equal(a.mem.hot, b.mem.hot)
    finally:
        a.close()
        b.close()


def test_cuda_graph_replay_equals_eager():
    w = get("dsa").scaled(R=3, groups=2, L_ctx=16384, steps=6)
    eager = Run(w)
    graph = Run(w)
    try:
        for t in range(w.steps):
            eager.step()
        torch.cuda.synchronize()
        # capture each step once, then replay it
        g_list = []
        s = torch.cuda.Stream()
        for t in range(w.steps):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(s):
                with torch.cuda.graph(g, stream=s):
                    graph.gpu_step(t)
            g_list.append(g)
        torch.cuda.synchronize()
        graph.hs.reset()
        graph.mem.hot.zero_()
        torch.cuda.synchronize()
        for t in range(w.steps):
            g_list[t].replay()
            graph.oracle_step(t)
        graph.compare()
        for a, _ in eager.groups:
            for x, y in zip(eager.hs.export_state(a), graph.hs.export_state(a)):
                np.testing.assert_array_equal(x, y)
    finally:
        eager.close()
        graph.close()


# ---------------------------------------------------------------------- #
def _largest_buffer(R, k, P_of, lookup):
    """The largest B that hisparse_init accepts for (R, k) (shared memory is
    the binding limit below the int16 LRU bound of 32767)."""
    def fits(B):
        mem = WorkloadMemory(R, 1, B, P_of(B), 16)
        try:
            hs = HiSparse(R, 1, k, B, P_of(B), 16, mem.layer_buffers(), lookup=lookup)
        except H.HiSparseError as e:
            assert e.code == H.EBOUND
            return False
        finally:
            mem.close()
        hs.close()
        return True
    lo, hi = k, 32767       # fits(lo) holds; find the last B that fits
    assert fits(lo)
    if fits(hi):
        return hi
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if fits(mid):
            lo = mid
        else:
            hi = mid
    return lo


@pytest.mark.parametrize("lookup", LOOKUPS)
@pytest.mark.parametrize("k", [64, 2048])
def test_largest_buffer_that_fits(k, lookup):
    """At the largest accepted B, from a full imported state (every slot
    occupied, LRU a random permutation), steps that mix hits and misses match
    the oracle; B + 1 is refused with EBOUND."""
    R = 2
    P_of = lambda B: 3 * B
    B = _largest_buffer(R, k, P_of, lookup)
    print(f"largest accepted B at k={k}, lookup={lookup}: {B}")
    P = P_of(B)
    rng = np.random.default_rng(B * 7 + k)
    mem, hs = _instance(R, k, B, P, lookup=lookup)
    o = OracleLayer(R, k, B, P, 16, host=mem.host_view(0))
    o.reset()
    sp = np.stack([rng.permutation(P)[:B] for _ in range(R)]).astype(np.int32)
    lru = np.stack([rng.permutation(B) for _ in range(R)]).astype(np.int16)
    pt = np.full((R, P), -1, np.int32)
    for r in range(R):
        pt[r, sp[r]] = np.arange(B, dtype=np.int32)
    assert hs.import_state(0, sp, lru, pt) == 0
    o.slot_pos[:] = sp
    o.lru[:] = lru
    o.page_table[:] = pt
    out = torch.empty((R, k), dtype=torch.int32, device="cuda")
    for t in range(6):
        sel = np.empty((R, k), np.int32)
        for r in range(R):
            resident = o.slot_pos[r][o.slot_pos[r] >= 0]
            absent = np.setdiff1d(np.arange(P, dtype=np.int32), resident)
            nh = int(rng.integers(0, k + 1))
            row = np.concatenate([rng.choice(resident, nh, replace=False),
                                  rng.choice(absent, k - nh, replace=False)])
            sel[r] = rng.permutation(row)
        hs.resolve(0, _dev(sel), out)
        oo, e = o.resolve(sel)
        assert e == 0
        np.testing.assert_array_equal(out.cpu().numpy(), oo)
    sp2, lru2, pt2, mc = hs.export_state(0)
    np.testing.assert_array_equal(sp2, o.slot_pos)
    np.testing.assert_array_equal(lru2, o.lru)
    np.testing.assert_array_equal(pt2, o.page_table)
    np.testing.assert_array_equal(mc, o.miss_count)
    np.testing.assert_array_equal(mem.hot[0].cpu().numpy()[:, :B], o.hot[:, :B])
    hs.close(); mem.close()
    if B < 32767:
        mem = WorkloadMemory(R, 1, B + 1, P_of(B + 1), 16)
        with pytest.raises(H.HiSparseError) as ei:
            HiSparse(R, 1, k, B + 1, P_of(B + 1), 16, mem.layer_buffers(), lookup=lookup)
        assert ei.value.code == H.EBOUND
        mem.close()


def test_num_reqs_zero_touches_nothing():
    """A graph padded down to no live request: every unit, slot vector and
    host row stays as it was (write-through included)."""
    run = Run(get("dsa").scaled(R=2, groups=1, L_ctx=8192, steps=3), num_reqs=0)
    try:
        for _ in range(3):
            run.step()
        run.compare()
        assert (run.out.cpu().numpy() == -7).all()
        sp, lru, pt, mc = run.hs.export_state(0)
        assert (sp == -1).all() and (pt == -1).all() and (mc == 0).all()
    finally:
        run.close()


@pytest.mark.parametrize("mode", ["group", "inline"])
def test_interleaved_rows_from_mirror(mode):
    """The HBM mirror of an interleaved pool has the pool's layout and strides."""
    _run_all(get("shared").scaled(R=2, groups=2, L_ctx=2048, steps=4), group=4, mirror=True,
             flags=H.FROM_MIRROR, inline_shared=mode == "inline")


def test_sm_copy_between_host_and_device():
    """hisparse_copy moves bytes exactly host->device, device->host and
    device->device, for sizes from one 16-byte chunk to several MB; bad
    sizes and alignments are refused."""
    from host_offload_serving_gb300.runtime import sm_copy
    rng = np.random.default_rng(5)
    for nb in (16, 4096 + 16, 299_168, 3 << 20):
        h = torch.from_numpy(rng.integers(0, 256, nb, dtype=np.uint8)).pin_memory()
        d = torch.empty(nb, dtype=torch.uint8, device="cuda")
        d2 = torch.empty(nb, dtype=torch.uint8, device="cuda")
        back = torch.zeros(nb, dtype=torch.uint8).pin_memory()
        sm_copy(d, h)
        sm_copy(d2, d)
        sm_copy(back, d2)
        torch.cuda.synchronize()
        assert torch.equal(back, h)
        assert torch.equal(d.cpu(), h)
    d = torch.empty(64, dtype=torch.uint8, device="cuda")
    assert H.hisparse_copy(d.data_ptr(), d.data_ptr() + 32, 24, None) == H.EINVAL
    assert H.hisparse_copy(d.data_ptr() + 8, d.data_ptr() + 32, 16, None) == H.EINVAL
    assert H.hisparse_copy(None, d.data_ptr(), 16, None) == H.EINVAL
    assert H.hisparse_copy(d.data_ptr(), d.data_ptr() + 32, 0, None) == H.OK
    torch.cuda.synchronize()


def _need_host_memory(nbytes):
    """Skip (with the reason) when the host cannot pin a pool of nbytes plus
    a margin; the pool is pinned memory, which the kernel cannot swap."""
    avail = 0
    with open("/proc/meminfo") as f:
        for line in f:
            if line.startswith("MemAvailable:"):
                avail = int(line.split()[1]) * 1024
    if avail < nbytes + (16 << 30):
        pytest.skip(f"needs {nbytes / 2**30:.1f} GiB of host memory plus 16 GiB, "
                    f"{avail / 2**30:.1f} GiB available")


@pytest.mark.parametrize("name", ["quest", "shared"])
def test_full_size_config(name):
    """The Quest-style and shared-index configs at full size (every request,
    layer and step; 53.7 GB and 77.3 GB host pools): slot vectors and miss
    counts equal the oracle's after every step; slot maps, LRU order, page
    tables, plans and every hot byte after the first and the last step; the
    prefill host rows are unchanged."""
    _need_host_memory(get(name).host_bytes())
    _run_all(get(name), every=10 ** 9)


def test_capacity_sweep_point_at_full_size():
    """The capacity-sweep point B=4096, f=0.87 (64 requests x 2 layers, 16
    steps) at the largest context whose pinned pool leaves 16 GiB of the
    host free: 1M positions (154.6 GB) on a host like the bench's, else 512K
    or 256K.  Slot vectors and miss counts after every step; the full state and
    every hot byte after the first and the last; the prefill rows at the end."""
    avail = 0
    with open("/proc/meminfo") as f:
        for line in f:
            if line.startswith("MemAvailable:"):
                avail = int(line.split()[1]) * 1024
    w = None
    for L in (1048576, 524288, 262144):
        cand = sweep_workload(4096, 0.87, L_ctx=L)
        if avail >= cand.host_bytes() + (16 << 30):
            w = cand
            break
    if w is None:
        pytest.skip(f"no sweep context fits {avail / 2**30:.1f} GiB of available host memory")
    print(f"capacity sweep at L_ctx={w.L_ctx} ({w.host_bytes() / 1e9:.1f} GB pool)")
    run = Run(w)
    try:
        for t in range(w.steps):
            run.step()
            if t == 0:
                run.compare(check_prefill=False)
            elif t == w.steps - 1:
                run.compare(check_prefill=True)
            else:
                run.compare_light()
    finally:
        run.close()


def test_graph_with_host_inputs_and_outputs_by_sm_copy():
    """A step graph that copies its selections up from pinned host memory and
    its slot vectors back with hisparse_copy (the end-to-end form): every
    step's host-side slot vector equals the oracle's."""
    from host_offload_serving_gb300.runtime import sm_copy
    from workload.traces import layer_traces
    w = get("tiny").scaled(steps=12)
    mem = WorkloadMemory(w.R, w.L, w.B, w.P, w.rec)
    from workload import records as REC
    REC.fill_host_pool(w, mem.geometry)
    hs = HiSparse(w.R, w.L, w.k, w.B, w.P, w.rec, mem.layer_buffers())
    o = OracleLayer(w.R, w.k, w.B, w.P, w.rec, host=mem.host_view(0))
    o.reset()
    sel, _ = layer_traces(w, 0)
    h_sel = torch.from_numpy(np.ascontiguousarray(sel)).pin_memory()        # [T][R][k]
    h_out = torch.full((w.steps, w.R, w.k), -7, dtype=torch.int32).pin_memory()
    d_sel = torch.empty((w.R, w.k), dtype=torch.int32, device="cuda")
    d_out = torch.empty((w.R, w.k), dtype=torch.int32, device="cuda")
    cap = torch.cuda.Stream()
    graphs = []
    for t in range(w.steps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                s = torch.cuda.current_stream()
                sm_copy(d_sel, h_sel[t], stream=s)
                hs.resolve(0, d_sel, d_out, stream=s)
                sm_copy(h_out[t], d_out, stream=s)
        graphs.append(g)
    torch.cuda.synchronize()
    for t in range(w.steps):
        graphs[t].replay()
        ref, e = o.resolve(sel[t])
        assert e == 0
        torch.cuda.synchronize()
        np.testing.assert_array_equal(h_out[t].numpy(), ref)
    assert np.array_equal(mem.hot[0].cpu().numpy(), o.hot)
    hs.close(); mem.close()


# ---------------------------------------------------------------------- #
# Short requests: growth by the previous token, lookup by position         #
# ---------------------------------------------------------------------- #
@pytest.mark.parametrize("cs", [0, 1, 3])
@pytest.mark.parametrize("shared", ["none", "group", "inline"])
def test_short_requests_mixed_batch(cs, shared):
    """A batch of short requests (admitted with their tokens preloaded, then
    grown by one token per step), requests that outgrow B during the run, and
    long requests, through the fused write-through with per-request sequence
    lengths: every step's slot vectors, slot maps, LRU orders, page tables,
    miss counts, plans, hot bytes of every layer and written-back host rows
    equal the oracle's."""
    R, k, B, rec, steps = 6, 64, 256, 64, 10
    lens0 = np.array([40, 200, 250, 600, 1000, 253], np.int32)
    P = int(lens0.max()) + steps
    L = 1 if shared == "none" else 3
    anchor_of = [-1] + [0] * (L - 1)
    rng = np.random.default_rng(17 + cs)
    mem = WorkloadMemory(R, L, B, P, rec)
    for l in range(L):
        mem.host_view(l)[:] = rng.integers(0, 256, size=(R, P, rec), dtype=np.uint8)
    hs = HiSparse(R, L, k, B, P, rec, mem.layer_buffers(), anchor_of=anchor_of,
                  ctas_per_request=cs)
    orc = []
    for l in range(L):
        o = OracleLayer(R, k, B, P, rec, host_split=0, metadata=l == 0)
        o.host_tail[:] = mem.host_view(l)
        orc.append(o)
    orc[0].reset()
    short0 = [r for r in range(R) if lens0[r] + 1 <= B]
    reqs = _dev(np.arange(R, dtype=np.int32))
    pre = np.where(lens0 + 1 <= B, lens0, 0).astype(np.int32)
    hs.admit(-1, reqs, _dev(pre))
    for r in range(R):
        orc[0].admit(r, int(pre[r]))
        for l in range(1, L):
            orc[l].preload_bytes(r, int(pre[r]))
    out = torch.empty((R, k), dtype=torch.int32, device="cuda")
    try:
        for t in range(steps):
            seq = lens0 + t + 1
            newest = lens0 + t
            prev = (newest - 1) if t > 0 else np.full(R, -1, np.int32)
            new_rows = rng.integers(0, 256, size=(L, R, rec), dtype=np.uint8)
            sel = np.full((R, k), -1, np.int32)
            for r in range(R):
                m = min(k - 2, int(seq[r]))
                pick = rng.choice(int(seq[r]), size=m, replace=False)
                if t > 0 and prev[r] not in pick:
                    pick[0] = prev[r]              # the local window: last token again
                sel[r, :m] = pick
            sel[1, 5] = sel[1, 6]                  # a repeat (short request: not an error)
            d_new = _dev(new_rows, torch.uint8)
            d_prev = _dev(prev.astype(np.int32))
            flags = H.WITH_SHARED if shared == "inline" else (H.RECORD_PLAN if L > 1 else 0)
            for l in range(1, L):
                if shared == "inline":
                    hs.writeback(l, d_prev, new_rows=d_new[l])
            hs.resolve_ex(0, _dev(sel), out, newest=_dev(newest.astype(np.int32)),
                          prev_pos=d_prev, new_rows=d_new[0], flags=flags,
                          seq_lens=_dev(seq.astype(np.int32)))
            if shared == "group":
                for l in range(1, L):
                    hs.writeback(l, d_prev, new_rows=d_new[l])
                hs.prefetch_plan(0, -1)
            # oracle: write-backs, new tokens, the step, the shared layers' bytes
            for l in range(L):
                if t > 0:
                    orc[l].writeback(prev)
                orc[l].set_newest_rows(new_rows[l])
            oo, e = orc[0].resolve_with_seq_lens(sel, newest, prev, seq)
            for l in range(1, L):
                orc[0].replay_into(orc[l])
            torch.cuda.synchronize()
            np.testing.assert_array_equal(out.cpu().numpy(), oo, err_msg=f"out step {t}")
            sp, lru, pt, mc = hs.export_state(0)
            np.testing.assert_array_equal(sp, orc[0].slot_pos, err_msg=f"slot_pos step {t}")
            np.testing.assert_array_equal(lru, orc[0].lru, err_msg=f"lru step {t}")
            np.testing.assert_array_equal(pt, orc[0].page_table, err_msg=f"page table step {t}")
            np.testing.assert_array_equal(mc, orc[0].miss_count, err_msg=f"misses step {t}")
            if shared == "group":
                c, pp, ps = hs.export_plan(0)
                for r in range(R):
                    assert list(zip(pp[r, :c[r]], ps[r, :c[r]])) == list(zip(
                        orc[0].plan_pos[r, :orc[0].plan_count[r]],
                        orc[0].plan_slot[r, :orc[0].plan_count[r]])), f"plan {r} step {t}"
            hot = mem.hot.cpu().numpy()
            for l in range(L):
                np.testing.assert_array_equal(hot[l], orc[l].hot, err_msg=f"hot {l} step {t}")
                np.testing.assert_array_equal(mem.host_view(l), orc[l].host_tail,
                                              err_msg=f"host rows {l} step {t}")
            flags_, ue = hs.status()
            np.testing.assert_array_equal(ue[0], orc[0].unit_err, err_msg=f"unit errors {t}")
        # the short requests took the short path throughout, with one growth per step
        sp = hs.export_state(0)[0]
        for r in short0:
            n = min(int(lens0[r]) + steps - 1, B)
            if lens0[r] + steps <= B:
                assert sp[r, :n].tolist() == list(range(n)), f"request {r} not in order"
    finally:
        hs.close()
        mem.close()


def test_short_workload_full_size_every_step():
    """8 requests x 4 layers with 3K-position contexts and B=4096, admitted
    with their prefill preloaded: every step takes the short path (growth by
    the previous token, lookup by position), write-through fused."""
    _run_all(get("short"))


@pytest.mark.parametrize("cs", [1, 3])
def test_short_workload_crossing_the_buffer(cs):
    """Contexts that outgrow B during the run: the short path until seq_len
    exceeds B, the general resolve after, every step compared."""
    _run_all(get("short").scaled(R=3, groups=2, L_ctx=1020, k=256, B=1024, steps=10,
                                 W_loc=16), ctas_per_request=cs)


def test_short_requests_rejected_by_the_hash_lookup():
    R, k, B, P = 2, 8, 16, 64
    mem, hs = _instance(R, k, B, P, lookup=H.LOOKUP_HASH)
    out = torch.empty((R, k), dtype=torch.int32, device="cuda")
    sel = _dev(np.array([[1, 2, 3, 4, 5, 6, 7, 8]] * R, np.int32))
    with pytest.raises(H.HiSparseError) as ei:
        hs.resolve_ex(0, sel, out, seq_lens=_dev(np.array([9, 9], np.int32)))
    assert ei.value.code == H.EINVAL
    hs.close(); mem.close()


@pytest.mark.parametrize("opt", ["resident", "union", "blocks"])
def test_short_requests_with_extended_options(opt):
    """Short and long requests in one batch with the other options of the
    general RESOLVE: a resident block table (resident rows come first on the
    short path too), union verify rows (repeats resolve once on the general
    path and are simply looked up on the short one), and block-id selections
    expanded in the kernel."""
    from oracle.tiny import expand_blocks
    R, k, B, rec, steps, bt = 4, 64, 128, 32, 8, 4
    lens0 = np.array([20, 100, 300, 121], np.int32)   # short, short, long, crossing
    P = int(lens0.max()) + steps
    rng = np.random.default_rng(31)
    mem = WorkloadMemory(R, 1, B, P, rec)
    mem.host_view(0)[:] = rng.integers(0, 256, size=(R, P, rec), dtype=np.uint8)
    hs = HiSparse(R, 1, k, B, P, rec, mem.layer_buffers())
    o = OracleLayer(R, k, B, P, rec, host_split=0)
    o.host_tail[:] = mem.host_view(0)
    o.reset()
    pre = np.where(lens0 + 1 <= B, lens0, 0).astype(np.int32)
    hs.admit(0, _dev(np.arange(R, dtype=np.int32)), _dev(pre))
    for r in range(R):
        o.admit(r, int(pre[r]))
    out = torch.empty((R, k), dtype=torch.int32, device="cuda")
    blocks = None
    if opt == "resident":
        blocks = np.full((R, P // 16 + 1), -1, np.int32)
        blocks[0, 0] = 5        # positions 0..15 of request 0 resident
        blocks[2, 3] = 9        # positions 48..63 of request 2 resident
    try:
        for t in range(steps):
            seq = lens0 + t + 1
            newest = lens0 + t
            prev = (newest - 1) if t > 0 else np.full(R, -1, np.int32)
            new_rows = rng.integers(0, 256, size=(R, rec), dtype=np.uint8)
            if opt == "blocks":
                kb = k // bt
                sel_gpu = np.full((R, kb), -1, np.int32)
                for r in range(R):
                    nb = min(kb, int(seq[r]) // bt)
                    sel_gpu[r, :nb] = rng.choice(int(seq[r]) // bt, size=nb, replace=False)
                sel = np.array([expand_blocks(row.tolist(), bt) for row in sel_gpu], np.int32)
            else:
                sel = np.full((R, k), -1, np.int32)
                for r in range(R):
                    m = min(k, int(seq[r]))
                    sel[r, :m] = rng.choice(int(seq[r]), size=m, replace=False)
                if opt == "union":
                    sel[:, k // 2:] = sel[:, :k // 2]   # a second verify row repeating the first
                sel_gpu = sel
            flags = H.UNION if opt == "union" else 0
            hs.resolve_ex(0, _dev(sel_gpu), out, newest=_dev(newest.astype(np.int32)),
                          prev_pos=_dev(prev.astype(np.int32)), new_rows=_dev(new_rows, torch.uint8),
                          res_blocks=None if blocks is None else _dev(blocks),
                          res_block_tokens=16 if blocks is not None else 0,
                          sel_block_tokens=bt if opt == "blocks" else 1, flags=flags,
                          seq_lens=_dev(seq.astype(np.int32)))
            if t > 0:
                o.writeback(prev)
            o.set_newest_rows(new_rows)
            oo, _ = o.resolve_with_seq_lens(sel, newest, prev, seq, res_blocks=blocks,
                                            res_tok=16, union=opt == "union")
            torch.cuda.synchronize()
            np.testing.assert_array_equal(out.cpu().numpy(), oo, err_msg=f"out step {t}")
            sp, lru, pt, mc = hs.export_state(0)
            np.testing.assert_array_equal(sp, o.slot_pos, err_msg=f"slot_pos step {t}")
            np.testing.assert_array_equal(lru, o.lru, err_msg=f"lru step {t}")
            np.testing.assert_array_equal(pt, o.page_table, err_msg=f"page table step {t}")
            np.testing.assert_array_equal(mc, o.miss_count, err_msg=f"misses step {t}")
            np.testing.assert_array_equal(mem.hot[0].cpu().numpy(), o.hot, err_msg=f"hot step {t}")
            np.testing.assert_array_equal(mem.host_view(0), o.host_tail, err_msg=f"host step {t}")
            flags_, ue = hs.status()
            np.testing.assert_array_equal(ue[0], o.unit_err, err_msg=f"unit errors {t}")
    finally:
        hs.close()
        mem.close()
