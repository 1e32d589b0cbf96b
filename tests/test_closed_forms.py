"""The pages' capacity and IO arithmetic, restated as closed forms.

gentlecold.top "HiSparse 深度解析" §2.3 (per-token IO), §3.1 (bounded
occupancy N_batch*N_l*B*W_KV*s instead of N_batch*N_l*L_ctx*W_KV*s) and §3.4
(GLM-5.1 at 128K: 13.09 GB per request, about 0.4 GB at B=4096).
"""
from workload import WORKLOADS


def occupancy(n_batch, n_layers, slots, w_kv, s):
    return n_batch * n_layers * slots * w_kv * s


def test_bounded_occupancy_glm51():
    full = 13.09e9                       # GB per request at 128K (the page's figure)
    per_slot = full / 131072             # bytes per position across layers
    assert abs(per_slot * 4096 / 1e9 - 0.409) < 0.001    # "约 0.4 GB"
    assert 131072 // 4096 == 32                           # "约 30 倍"


def test_per_token_io():
    kv_per_token = 100e3                 # "每 token 跨层约 100 KB"
    k = 2048
    no_cache = kv_per_token * k
    assert abs(no_cache / 1e6 - 204.8) < 1e-9             # "约 200 MB"
    assert abs(no_cache / 30e-3 / 1e9 - 6.83) < 0.01      # "约 7 GB/s" at 30 ms TPOT
    assert abs(0.134 * no_cache / 1e6 - 27.4) < 0.1       # "约 27 MB" at 13.4% miss


def test_workload_hot_buffer_matches_formula():
    for w in WORKLOADS.values():
        assert w.hot_bytes() == occupancy(w.R, w.L, w.B + 1, w.rec, 1)
        assert w.host_bytes() == occupancy(w.R, w.L, w.P, w.rec, 1)
