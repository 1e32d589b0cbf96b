"""The seeded input generators: deterministic, well-formed, shaped as stated."""
import numpy as np
import pytest

from workload import get, WORKLOADS, sweep_workload
from workload.traces import unit_trace, zipf_cdf
from workload import records


def test_traces_are_deterministic_and_distinct_per_unit():
    w = get("tiny")
    a, na = unit_trace(w, 0, 0)
    b, nb = unit_trace(w, 0, 0)
    assert (a == b).all() and (na == nb).all()
    w2 = w.scaled(R=2)
    c, _ = unit_trace(w2, 0, 1)
    assert not (a == c).all()


@pytest.mark.parametrize("name", ["tiny", "quest"])
def test_trace_structure(name):
    w = get(name)
    sel, newest = unit_trace(w, 0, 0)
    assert sel.shape == (w.steps, w.k) and sel.dtype == np.int32
    for t in range(w.steps):
        s = sel[t]
        assert len(set(s.tolist())) == w.k                       # distinct
        assert s.min() >= 0 and s.max() < w.P
        mand = set(range(w.n_sink)) | set(range(w.L_ctx - w.W_loc, w.L_ctx)) if w.W_loc else set(range(w.n_sink))
        if t > 0 or w.step0 != "uniform":
            assert mand <= set(s.tolist())
    # reuse close to f: share of S_t found in S_{t-1}
    reuse = np.mean([len(set(sel[t]) & set(sel[t - 1])) / w.k for t in range(1, w.steps)])
    assert abs(reuse - w.f) < 0.05


def test_write_through_trace_has_newest_in_local_window():
    w = get("dsa").scaled(R=1, groups=1, L_ctx=8192, k=256, B=512, steps=6)
    sel, newest = unit_trace(w, 0, 0)
    for t in range(w.steps):
        assert newest[t] == w.L_ctx + t
        assert newest[t] in set(sel[t].tolist())
        assert sel[t].max() <= newest[t]                           # causal


def test_all_hit_trace_repeats_step0():
    w = sweep_workload(2048, 0.87, L_ctx=16384, all_hit=True).scaled(k=128, B=256, steps=4)
    sel, _ = unit_trace(w, 0, 0)
    assert all((sel[t] == sel[0]).all() for t in range(w.steps))


def test_zipf_cdf():
    c = zipf_cdf(4, 1.0)
    h = 1 + 1 / 2 + 1 / 3 + 1 / 4
    assert np.allclose(c, np.cumsum([1 / h, 1 / (2 * h), 1 / (3 * h), 1 / (4 * h)]))


def test_bf16_rounding():
    f = np.array([1.0, -2.5, 1.00390625, 1.01171875, 3.0e-3], np.float32)
    b = records.f32_to_bf16_rne(f)
    back = (b.astype(np.uint32) << 16).view(np.float32)
    assert back[0] == 1.0 and back[1] == -2.5
    assert back[2] == 1.0            # tie rounds to even
    assert back[3] == 1.015625       # tie rounds to even (up)
    assert abs(back[4] - 3.0e-3) / 3.0e-3 < 2 ** -8


def test_normal_table_moments():
    t = records.normal_table()
    v = (t.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert abs(v.mean()) < 1e-3 and abs(v.std() - 1.0) < 5e-3
    assert (np.diff(v) >= 0).all()


def test_records_deterministic_and_keyed():
    w = get("tiny")
    a = records.records(w, 0, 0, [0, 1, 4095])
    b = records.records(w, 0, 0, [0, 1, 4095])
    assert (a == b).all()
    assert not (a[0] == a[1]).all()
    c = records.records(w.scaled(R=2), 0, 1, [0])
    assert not (a[0] == c[0]).all()
    # pool fill == per-position fill
    pool = np.zeros((w.P, w.rec), np.uint8)
    records.fill(pool.ctypes.data, w.P, w.rec, w.rec, w.seed, 0, 0, 0)
    assert (pool[[0, 1, 4095]] == a).all()


def test_workload_sizes():
    dsa = WORKLOADS["dsa"]
    assert dsa.P == 131072 + 32
    assert abs(dsa.host_bytes() / 1e9 - 4.83) < 0.01
    assert WORKLOADS["shared"].anchor_of()[:5] == [-1, 0, 0, 0, -1]
    assert WORKLOADS["shared"].anchors() == [0, 4, 8, 12]


def test_short_workload_fits_the_short_path():
    """The short-request workload: every request's context fits the buffer
    for the whole run (seq_len = L_ctx + t + 1 <= B), every selection is a
    position below seq_len, and the newest position is selected (the local
    window), so every step of every unit takes the short path."""
    w = get("short")
    assert w.admit_preload and w.write_through
    assert w.L_ctx + w.steps <= w.B
    for r in range(2):
        sel, newest = unit_trace(w, 0, r)
        for t in range(w.steps):
            seq_len = w.L_ctx + t + 1
            assert newest[t] == seq_len - 1
            assert sel[t].min() >= 0 and sel[t].max() < seq_len
            assert newest[t] in set(sel[t].tolist())
