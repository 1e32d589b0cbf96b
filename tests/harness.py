"""Run a workload on the CUDA path and on the oracle side by side (GPU tests).

The GPU side goes only through the C ABI (``host_offload_serving_gb300``); the
oracle side is the plain C model (``oracle.coracle``).  They share the seeded
inputs from ``workload`` and nothing else.
"""
import numpy as np
import torch

from host_offload_serving_gb300 import hisparse as H
from host_offload_serving_gb300.runtime import HiSparse, WorkloadMemory, DecodeStep
from oracle.coracle import OracleLayer
from workload import records as REC
from workload.traces import all_traces


class Run:
    def __init__(self, w, flags=0, mirror=False, ctas_per_request=0, replay_ctas=0,
                 num_reqs=None, oracle_bytes=True, traces=None, lookup=0, pool_kind=H.HOST_PINNED,
                 fused=True, resident=None, group=1, group_replay=True, inline_shared=False,
                 l2_persist=0):
        """``resident`` = (int32 [steps][R][nblk] block tables, tokens per
        block) runs every anchor through the three-tier resolve, with the
        table of step t in place before step t."""
        self.w = w
        self.flags = flags
        self.lookup = lookup
        dev = torch.device("cuda", 0)
        self.mem = WorkloadMemory(w.R, w.L, w.B, w.P, w.rec, mirror=mirror, pool_kind=pool_kind,
                                  group=group)
        REC.fill_host_pool(w, self.mem.geometry)
        if mirror:
            self.mem.fill_mirror()
        self.hs = HiSparse(w.R, w.L, w.k, w.B, w.P, w.rec, self.mem.layer_buffers(),
                           anchor_of=w.anchor_of(), ctas_per_request=ctas_per_request,
                           replay_ctas=replay_ctas, lookup=lookup)
        if l2_persist:
            self.hs.set_l2_persisting(l2_persist)
        anchor_of = w.anchor_of()
        self.groups = [(a, [l for l in range(w.L) if anchor_of[l] == a]) for a in w.anchors()]
        tr = traces if traces is not None else all_traces(w)
        self.sel_np = np.stack([tr[a][0] for a, _ in self.groups], axis=1)  # [T][G][R][k]
        self.sel_gpu_np = self.sel_np
        bt = w.sel_block_tokens
        if bt > 1:   # the GPU reads block ids; the oracle gets the positions
            from oracle.tiny import expand_blocks
            blk = self.sel_np
            pos = (blk[..., None].astype(np.int64) * bt + np.arange(bt)).reshape(*blk.shape[:-1], -1)
            pos = np.where(np.repeat(blk == -1, bt, axis=-1), -1, pos).astype(np.int32)
            assert pos[0, 0, 0].tolist() == expand_blocks(blk[0, 0, 0].tolist(), bt)
            self.sel_np = pos
        self.newest_np = tr[self.groups[0][0]][1] if w.write_through else None  # [T][R]
        self.sel = torch.from_numpy(self.sel_gpu_np).to(dev)
        self.newest = torch.from_numpy(self.newest_np).to(dev) if w.write_through else None
        self.new_rows_np = REC.new_token_records(w)                       # [T][L][R][rec]
        self.new_rows = torch.from_numpy(self.new_rows_np).to(dev) if w.write_through else None
        if w.write_through:
            wb = np.full((w.steps, w.L, w.R), -1, np.int32)
            for t in range(1, w.steps):
                wb[t] = self.newest_np[t - 1][None, :]
            self.wb_np = wb
            self.wb = torch.from_numpy(wb).to(dev)
        self.out = torch.full((len(self.groups), w.R, w.k), -7, dtype=torch.int32, device=dev)
        self.nreq_val = w.R if num_reqs is None else num_reqs
        self.num_reqs = torch.tensor([self.nreq_val], dtype=torch.int32, device=dev)
        self.res_np = self.res_dev = None
        self.res_tok = 1
        if resident is not None:
            self.res_np, self.res_tok = resident
            self.res_dev = torch.from_numpy(np.ascontiguousarray(self.res_np[0])).to(dev)
        self.step_runner = DecodeStep(self.hs, self.mem, self.groups, flags=flags,
                                      num_reqs=self.num_reqs, fused=fused,
                                      resident=None if resident is None else
                                      (self.res_dev, self.res_tok), sel_block_tokens=bt,
                                      group_replay=group_replay, inline_shared=inline_shared)
        # oracle
        self.oracle = {}
        for l in range(w.L):
            is_anchor = anchor_of[l] < 0
            o = OracleLayer(w.R, w.k, w.B, w.P, w.rec, host=self.mem.host_view(l),
                            host_split=w.L_ctx, keep_bytes=oracle_bytes, metadata=is_anchor)
            if is_anchor:
                o.reset()
            self.oracle[l] = o
        self.oracle_out = np.full((len(self.groups), w.R, w.k), -7, np.int32)
        self.seq_np = self.seq = None
        if w.admit_preload:   # short requests: admitted with their prefill preloaded
            self.seq_np = (w.L_ctx + 1 + np.arange(w.steps, dtype=np.int32))[:, None].repeat(
                w.R, axis=1)                                               # [T][R]
            self.seq = torch.from_numpy(np.ascontiguousarray(self.seq_np)).to(dev)
            self.admit(list(range(w.R)), [w.L_ctx] * w.R)
        self.t = 0

    # ------------------------------------------------------------------ #
    def gpu_step(self, t):
        if self.res_dev is not None:
            self.res_dev.copy_(torch.from_numpy(np.ascontiguousarray(self.res_np[t])))
        self.step_runner.issue(self.sel[t], self.out,
                               newest=self.newest[t] if self.newest is not None else None,
                               wb_pos=self.wb[t] if (self.w.write_through and t > 0) else None,
                               new_rows=self.new_rows[t] if self.new_rows is not None else None,
                               seq_lens=self.seq[t] if self.seq is not None else None)

    def oracle_step(self, t):
        w = self.w
        nr = self.nreq_val
        io = not (self.flags & H.SKIP_IO)
        if w.write_through:
            for l in range(w.L):
                if t > 0:
                    self.oracle[l].writeback(self.wb_np[t, l], num_reqs=nr)
                # the write-back launch places the new token's KV in row B of
                # every live request
                self.oracle[l].set_newest_rows(self.new_rows_np[t, l], num_reqs=nr)
        for gi, (a, fl) in enumerate(self.groups):
            nw = self.newest_np[t] if self.newest_np is not None else None
            if self.seq_np is not None:
                prev = self.wb_np[t, a] if t > 0 else np.full(w.R, -1, np.int32)
                out, _ = self.oracle[a].resolve_with_seq_lens(
                    self.sel_np[t, gi], nw, prev, self.seq_np[t], num_reqs=nr, io=io,
                    res_blocks=None if self.res_np is None else self.res_np[t],
                    res_tok=self.res_tok, union=bool(self.flags & H.UNION))
            else:
                out, _ = self.oracle[a].resolve(self.sel_np[t, gi], nw, num_reqs=nr, io=io,
                                                res_blocks=None if self.res_np is None else
                                                self.res_np[t], res_tok=self.res_tok,
                                                union=bool(self.flags & H.UNION))
            self.oracle_out[gi, :nr] = out[:nr]
            for f in fl:
                self.oracle[a].replay_into(self.oracle[f], num_reqs=nr)

    def admit(self, reqs, preload):
        """Admit requests on every layer: GPU through hisparse_admit, oracle
        through its admission (anchors) and the lockstep bytes (shared)."""
        dev = self.out.device
        self.hs.admit(-1, torch.tensor(reqs, dtype=torch.int32, device=dev),
                      torch.tensor(preload, dtype=torch.int32, device=dev))
        anchor_of = self.w.anchor_of()
        for l, o in self.oracle.items():
            for r, n in zip(reqs, preload):
                if anchor_of[l] < 0:
                    o.admit(r, n)
                else:
                    o.preload_bytes(r, n)

    def step(self):
        self.gpu_step(self.t)
        self.oracle_step(self.t)
        self.t += 1

    # ------------------------------------------------------------------ #
    def compare_light(self):
        """Assert GPU == oracle on this step's slot vectors and miss counts
        (the per-step outputs; cheap enough for every step at full size)."""
        torch.cuda.synchronize()
        nr = self.nreq_val
        out = self.out.cpu().numpy()
        np.testing.assert_array_equal(out[:, :nr], self.oracle_out[:, :nr],
                                      err_msg=f"out slots after step {self.t - 1}")
        mcd = torch.empty(self.w.R, dtype=torch.int32, device=self.out.device)
        for a, _ in self.groups:
            self.hs.copy_miss_counts(a, mcd)
            mc = mcd.cpu().numpy()
            np.testing.assert_array_equal(mc[:nr], self.oracle[a].miss_count[:nr],
                                          err_msg=f"miss count {a} after step {self.t - 1}")

    def compare(self, check_bytes=True, check_page_table=True, check_prefill=True):
        """Assert GPU == oracle on every field of every layer (synchronises).

        The plan is compared in list order with the page-table lookup (which
        records it in list order) and as a set of (position, slot) pairs with
        the hash lookup (which records it in host-row order).  With
        ``check_prefill`` the host rows below L_ctx -- the rows the oracle
        reads from the same pool -- are also checked against a fresh
        generation of the records, so that a stray store into them cannot
        pass unseen by changing both sides' input."""
        torch.cuda.synchronize()
        w = self.w
        nr = self.nreq_val
        out = self.out.cpu().numpy()
        np.testing.assert_array_equal(out[:, :nr], self.oracle_out[:, :nr], err_msg="out slots")
        for a, fl in self.groups:
            sp, lru, pt, mc = self.hs.export_state(a)
            o = self.oracle[a]
            np.testing.assert_array_equal(sp, o.slot_pos, err_msg=f"slot_pos layer {a}")
            np.testing.assert_array_equal(lru, o.lru, err_msg=f"lru layer {a}")
            np.testing.assert_array_equal(mc[:nr], o.miss_count[:nr], err_msg=f"miss count {a}")
            if check_page_table:
                np.testing.assert_array_equal(pt, o.page_table, err_msg=f"page table {a}")
            if fl and not self.step_runner.inline_shared:  # the recorded plan
                c, pp, ps = self.hs.export_plan(a)
                in_order = self.lookup == H.LOOKUP_PAGE_TABLE
                for r in range(nr):
                    got = list(zip(pp[r, :c[r]].tolist(), ps[r, :c[r]].tolist()))
                    exp = list(zip(o.plan_pos[r, :o.plan_count[r]].tolist(),
                                   o.plan_slot[r, :o.plan_count[r]].tolist()))
                    if not in_order:
                        got, exp = sorted(got), sorted(exp)
                    assert got == exp, f"plan of layer {a} request {r}"
        if check_prefill:
            self.check_prefill_intact()
        if check_bytes:
            hot = self.mem.hot.cpu().numpy()
            for l in range(w.L):
                np.testing.assert_array_equal(hot[l], self.oracle[l].hot, err_msg=f"hot bytes {l}")
                if w.P > w.L_ctx:
                    tail = self.mem.host_view(l)[:, w.L_ctx:, :]
                    np.testing.assert_array_equal(tail, self.oracle[l].host_tail,
                                                  err_msg=f"host tail {l}")
        flags, ue = self.hs.status()
        assert flags == 0, f"status flags {flags}"

    def check_prefill_intact(self, chunk_rows=16384):
        """Host rows [0, L_ctx) of every (layer, request) equal a fresh
        generation of their records (``workload.records``), chunk by chunk."""
        w = self.w
        buf = np.empty((min(chunk_rows, w.L_ctx), w.rec), np.uint8)
        for l in range(w.L):
            view = self.mem.host_view(l)
            for r in range(w.R):
                for p0 in range(0, w.L_ctx, chunk_rows):
                    n = min(chunk_rows, w.L_ctx - p0)
                    REC.fill(buf.ctypes.data, n, w.rec, w.rec, w.seed, l, r, p0)
                    if not np.array_equal(view[r, p0:p0 + n], buf[:n]):
                        bad = np.nonzero((view[r, p0:p0 + n] != buf[:n]).any(axis=1))[0]
                        raise AssertionError(f"prefill host rows changed: layer {l} request {r} "
                                             f"rows {(bad[:8] + p0).tolist()}")

    def close(self):
        self.hs.close()
        self.mem.close()
