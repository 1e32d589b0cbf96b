"""Host-side orchestration of the HiSparse hot path (memory, streams, events).

``HostPool``   pinned, device-mapped host memory from ``hisparse_host_alloc``.
``HiSparse``   one library instance: holds the handle, checks every return code.
``DecodeStep`` issues one decode step over all layers the way the pages order
               it (gentlecold.top "HiSparse 深度解析" §3.4 write-through, §3.6 and
               §5.6 plan-then-IO prefetch; docs.vllm.ai "HiSparse local KV
               offload architecture", performance invariants):
                 backup stream : write-through of the previous token, event
                 compute stream: wait for the write-through, place the new
                                 token's KV in row B, RESOLVE each anchor
                                 (recording its plan when it has followers)
                 side stream   : after each anchor, replay its plan into its
                                 followers (one launch for all of them, or one
                                 per follower), events per follower
               or, with ``inline_shared``, the followers filled inside the
               anchor's RESOLVE launch.  No call in a step allocates or reads
               device values on the host, so a whole step can be captured in a
               CUDA graph.
``sm_copy``    host <-> HBM copies by SM threads (``hisparse_copy``).

torch is used for device memory, streams, events and graphs only; every byte
and index of the hot path is produced by the kernels in ``libhisparse.so``.
"""
import ctypes

import numpy as np
import torch

from . import hisparse as H


class HostPool:
    """Pinned + mapped host memory of exactly ``nbytes`` (freed by ``close``)."""

    def __init__(self, nbytes, kind=H.HOST_PINNED):
        rc, ptr = H.hisparse_host_alloc_kind(int(nbytes), kind)
        H.check(rc, f"hisparse_host_alloc_kind({nbytes}, {kind})")
        self.ptr = ptr
        self.nbytes = int(nbytes)

    def hugepage_fraction(self):
        rc, huge = H.hisparse_host_hugepage_bytes(self.ptr, self.nbytes)
        return huge / self.nbytes if rc == H.OK and self.nbytes else 0.0

    def numpy(self):
        buf = (ctypes.c_uint8 * self.nbytes).from_address(self.ptr)
        return np.ctypeslib.as_array(buf)

    def close(self):
        if self.ptr:
            H.check(H.hisparse_host_free(self.ptr), "hisparse_host_free")
            self.ptr = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s):
    if s is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def sm_copy(dst, src, stream=None):
    """Copy tensor ``src`` into tensor ``dst`` (same byte size, a multiple of
    16) with SM threads (``hisparse_copy``); either may be pinned host memory."""
    nb = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nb:
        raise ValueError("sm_copy: sizes differ")
    H.check(H.hisparse_copy(_ptr(dst), _ptr(src), nb, _stream(stream)), "hisparse_copy")


class HiSparse:
    """One instance of the C library (R requests, L layers, k, B, P, record)."""

    def __init__(self, R, L, k, B, P, rec, layers, anchor_of=None, ctas_per_request=0,
                 replay_ctas=0, lookup=0):
        self.R, self.L, self.k, self.B, self.P, self.rec = R, L, k, B, P, rec
        self.anchor_of = list(anchor_of) if anchor_of is not None else [-1] * L
        self._anchor_arr = (ctypes.c_int32 * L)(*self.anchor_of)
        cfg = H.Config(R, L, k, B, P, rec, ctas_per_request, replay_ctas, lookup,
                       ctypes.cast(self._anchor_arr, ctypes.c_void_p))
        rc, h = H.hisparse_init(cfg, layers)
        H.check(rc, "hisparse_init")
        self.h = h

    # ---- launches (asynchronous, graph-capturable) ----
    def resolve(self, layer, sel, out, num_reqs=None, newest=None, flags=0, stream=None):
        H.check(H.hisparse_resolve(self.h, layer, _ptr(sel), _ptr(num_reqs), _ptr(newest),
                                   _ptr(out), flags, _stream(stream)), "hisparse_resolve")

    def resolve_step(self, layer, sel, out, num_reqs=None, newest=None, prev_pos=None,
                     new_rows=None, flags=0, stream=None):
        H.check(H.hisparse_resolve_step(self.h, layer, _ptr(sel), _ptr(num_reqs), _ptr(newest),
                                        _ptr(prev_pos), _ptr(new_rows), _ptr(out), flags,
                                        _stream(stream)), "hisparse_resolve_step")

    def resolve_resident(self, layer, sel, out, res_blocks, res_block_tokens, num_reqs=None,
                         newest=None, prev_pos=None, new_rows=None, flags=0, stream=None):
        """Three-tier RESOLVE: ``res_blocks`` is a device int32 [R][max_blocks]
        resident block table (-1 = not resident), ``res_block_tokens``
        positions per block."""
        H.check(H.hisparse_resolve_resident(self.h, layer, _ptr(sel), _ptr(num_reqs),
                                            _ptr(newest), _ptr(prev_pos), _ptr(new_rows),
                                            _ptr(res_blocks), int(res_blocks.shape[1]),
                                            int(res_block_tokens), _ptr(out), flags,
                                            _stream(stream)), "hisparse_resolve_resident")

    def resolve_ex(self, layer, sel, out, num_reqs=None, newest=None, prev_pos=None,
                   new_rows=None, res_blocks=None, res_block_tokens=0, sel_block_tokens=1,
                   flags=0, stream=None, seq_lens=None):
        """The general RESOLVE (``hisparse_resolve_ex``): fused write-through,
        resident tier, block-id selections and short requests (``seq_lens``,
        device int32 [R]), each optional."""
        o = H.ResolveOptions(_ptr(prev_pos), _ptr(new_rows), _ptr(res_blocks),
                             int(res_blocks.shape[1]) if res_blocks is not None else 0,
                             int(res_block_tokens), int(sel_block_tokens), _ptr(seq_lens))
        H.check(H.hisparse_resolve_ex(self.h, layer, _ptr(sel), _ptr(num_reqs), _ptr(newest), o,
                                      _ptr(out), flags, _stream(stream)), "hisparse_resolve_ex")

    def admit(self, layer, reqs, preload=None, stream=None):
        """Reset the listed requests (device int32 [n]) of ``layer`` (-1: all)
        and preload the first ``preload[i]`` positions of each (device int32
        [n], or None for none)."""
        H.check(H.hisparse_admit(self.h, layer, _ptr(reqs), int(reqs.numel()), _ptr(preload),
                                 _stream(stream)), "hisparse_admit")

    def writeback(self, layer, pos, num_reqs=None, stream=None, new_rows=None):
        H.check(H.hisparse_writeback(self.h, layer, _ptr(pos), _ptr(new_rows), _ptr(num_reqs),
                                     _stream(stream)), "hisparse_writeback")

    def prefetch_plan(self, anchor, follower, num_reqs=None, stream=None):
        H.check(H.hisparse_prefetch_plan(self.h, anchor, follower, _ptr(num_reqs),
                                         _stream(stream)), "hisparse_prefetch_plan")

    def copy_miss_counts(self, layer, dst, stream=None):
        H.check(H.hisparse_copy_miss_counts(self.h, layer, _ptr(dst), _stream(stream)),
                "hisparse_copy_miss_counts")

    def reset(self, layer=-1, stream=None):
        H.check(H.hisparse_reset(self.h, layer, _stream(stream)), "hisparse_reset")

    # ---- synchronous queries ----
    def status(self):
        ue = np.zeros((self.L, self.R), np.int32)
        rc, flags = H.hisparse_get_status(self.h, ue.ctypes.data)
        H.check(rc, "hisparse_get_status")
        return flags, ue

    def export_state(self, layer):
        sp = np.empty((self.R, self.B), np.int32)
        lru = np.empty((self.R, self.B), np.int16)
        pt = np.empty((self.R, self.P), np.int32)
        mc = np.empty(self.R, np.int32)
        H.check(H.hisparse_export_state(self.h, layer, sp.ctypes.data, lru.ctypes.data,
                                        pt.ctypes.data, mc.ctypes.data), "hisparse_export_state")
        return sp, lru, pt, mc

    def import_state(self, layer, slot_pos, lru, page_table, miss_counts=None):
        """Returns the C return code (validation failures are EINVAL)."""
        sp = np.ascontiguousarray(slot_pos, np.int32)
        lr = np.ascontiguousarray(lru, np.int16)
        pt = np.ascontiguousarray(page_table, np.int32)
        mc = None if miss_counts is None else np.ascontiguousarray(miss_counts, np.int32)
        return H.hisparse_import_state(self.h, layer, sp.ctypes.data, lr.ctypes.data,
                                       pt.ctypes.data, None if mc is None else mc.ctypes.data)

    def export_plan(self, layer):
        c = np.empty(self.R, np.int32)
        p = np.empty((self.R, self.k), np.int32)
        s = np.empty((self.R, self.k), np.int32)
        H.check(H.hisparse_export_plan(self.h, layer, c.ctypes.data, p.ctypes.data, s.ctypes.data),
                "hisparse_export_plan")
        return c, p, s

    def set_l2_persisting(self, nbytes):
        """Keep the RESOLVE layers' page tables in L2 (``hisparse_set_l2_persisting``;
        0 turns it off)."""
        H.check(H.hisparse_set_l2_persisting(self.h, int(nbytes)), "hisparse_set_l2_persisting")

    def info(self):
        rc, info = H.hisparse_get_info(self.h)
        H.check(rc, "hisparse_get_info")
        return {f: getattr(info, f) for f, _ in H.Info._fields_}

    def close(self):
        if self.h:
            H.check(H.hisparse_destroy(self.h), "hisparse_destroy")
            self.h = None


class WorkloadMemory:
    """Host pools, hot buffers and optional HBM mirrors for a workload.

    Host pools: one pinned allocation.  With ``group = 1`` layer l's rows are
    ``[R][P][rec]`` at ``pool + l*layer_stride``.  With ``group = m > 1``
    (shared-index groups of m layers: an anchor and its followers) the m
    layers of a group are interleaved row by row, ``[L/m][R][P][m][rec]``, so
    a position's records for the whole group are adjacent and a follower's
    replay reads the same host pages as its anchor's fetch just did.  The
    RESOLVE calls see only each layer's base and strides.
    Hot buffer of layer l: ``hot[l]`` (uint8 [R][B+1][rec], device).
    """

    def __init__(self, R, L, B, P, rec, device="cuda", mirror=False, pool_kind=H.HOST_PINNED,
                 group=1):
        if L % group:
            raise ValueError("the layer count must be a multiple of the group size")
        self.R, self.L, self.B, self.P, self.rec, self.group = R, L, B, P, rec, group
        self.req_stride = P * rec * group
        self.row_stride = rec * group
        self.layer_stride = R * P * rec            # bytes of one layer's rows
        self.pool = HostPool(L * self.layer_stride, kind=pool_kind)
        self.hot = torch.zeros((L, R, B + 1, rec), dtype=torch.uint8, device=device)
        self.mirror = None
        if mirror:   # byte for byte the pool's layout, so it shares the pool's strides
            self.mirror = torch.empty(L * self.layer_stride, dtype=torch.uint8, device=device)

    def layer_offset(self, layer):
        """Byte offset of layer ``layer``'s row (0, 0) in the pool."""
        g, j = divmod(layer, self.group)
        return g * self.group * self.layer_stride + j * self.rec

    def geometry(self, layer):
        """(address of row (0, 0), request stride, row stride) of a layer."""
        return self.pool.ptr + self.layer_offset(layer), self.req_stride, self.row_stride

    def host_view(self, layer):
        """numpy uint8 [R][P][rec] view of one layer's host rows."""
        a = self.pool.numpy()
        return np.lib.stride_tricks.as_strided(
            a[self.layer_offset(layer):], shape=(self.R, self.P, self.rec),
            strides=(self.req_stride, self.row_stride, 1), writeable=True)

    def layer_buffers(self):
        out = []
        for l in range(self.L):
            base, rs, ws = self.geometry(l)
            out.append(H.LayerBuffers(
                base, rs, ws, self.hot[l].data_ptr(), (self.B + 1) * self.rec, self.rec,
                self.mirror.data_ptr() + self.layer_offset(l) if self.mirror is not None else None))
        return out

    def fill_mirror(self):
        """Copy the host pool into the HBM mirror (pinned -> device)."""
        self.mirror.copy_(torch.from_numpy(self.pool.numpy()[:self.mirror.numel()]),
                          non_blocking=False)

    def close(self):
        self.pool.close()


class DecodeStep:
    """Issue decode steps over all layers with the stream/event order of the pages.

    ``groups`` is a list of (anchor layer, [follower layers]).  Per step t the
    caller provides device tensors: ``sel[t]`` int32 [Lr][R][k] (Lr = anchors),
    ``newest[t]`` int32 [R] or None, ``wb_pos[t]`` int32 [L][R] or None (rows to
    write back first), ``new_rows[t]`` uint8 [L][R][rec] or None (the new
    token's KV, placed in row B), and ``out`` int32 [Lr][R][k] receives the slot
    vectors.

    ``resident`` (optional) = (device int32 [R][max_blocks] resident block
    table, tokens per block) resolves every anchor with the resident tier
    first; ``sel_block_tokens`` > 1 means ``sel`` holds block ids of that many
    positions each (both through ``hisparse_resolve_ex``).

    ``group_replay=True`` (default) fills all of an anchor's shared-index
    layers with one ``hisparse_prefetch_plan(anchor, -1)`` launch, reading
    each plan record's rows for all of them back to back; ``False`` issues one
    replay per layer, as the pages do.

    ``inline_shared=True`` fills an anchor's shared-index layers inside the
    anchor's own RESOLVE launch (``HISPARSE_WITH_SHARED``) instead of replaying
    its plan on the side stream; their write-backs then go first, on the
    compute stream.

    ``fused=True`` (default) writes each anchor's previous token through, and
    installs its new token, inside that anchor's RESOLVE launch
    (``hisparse_resolve_step``); shared-index layers get a write-back launch on
    the side stream ahead of their replays.  ``fused=False`` issues one
    ``hisparse_writeback`` for every layer on a backup stream first, as the
    pages describe (gentlecold.top "HiSparse 深度解析" §5.4).
    """

    def __init__(self, hs, mem, groups, flags=0, num_reqs=None, fused=True, resident=None,
                 sel_block_tokens=1, group_replay=True, inline_shared=False):
        self.hs, self.mem, self.groups = hs, mem, groups
        self.group_replay = group_replay
        self.inline_shared = inline_shared
        self.flags = flags
        self.num_reqs = num_reqs
        self.fused = fused
        self.resident = resident    # (device int32 [R][max_blocks], tokens per block) or None
        self.sel_block_tokens = sel_block_tokens
        self.compute = torch.cuda.Stream()
        self.backup = torch.cuda.Stream()
        self.side = torch.cuda.Stream()
        self.ev_wb = torch.cuda.Event()
        self.ev_anchor = [torch.cuda.Event() for _ in groups]
        self.ev_follow = [[torch.cuda.Event() for _ in f] for _, f in groups]
        self.ev_step_start = torch.cuda.Event()
        self.ev_side_done = torch.cuda.Event()
        self._nopos = torch.full((hs.L, hs.R), -1, dtype=torch.int32, device=mem.hot.device)

    def _no_pos(self):
        return self._nopos

    def issue(self, sel, out, newest=None, wb_pos=None, new_rows=None, seq_lens=None):
        """Enqueue one step on the instance's streams (returns immediately).
        ``seq_lens`` (device int32 [R], optional): each request's positions so
        far; requests whose length fits the buffer take the short path
        (``hisparse_resolve_options.d_seq_lens``)."""
        hs = self.hs
        cur = torch.cuda.current_stream()
        self.ev_step_start.record(cur)
        self.compute.wait_event(self.ev_step_start)
        through = wb_pos is not None or new_rows is not None
        pos = wb_pos if wb_pos is not None else self._no_pos()
        if through and not self.fused:
            # one launch writes row B of every layer through to the host and
            # then places the new token's KV there ([DD] §3.4 step 4)
            self.backup.wait_event(self.ev_step_start)
            hs.writeback(-1, pos, self.num_reqs, stream=self.backup, new_rows=new_rows)
            self.ev_wb.record(self.backup)
            self.compute.wait_event(self.ev_wb)
        for gi, (anchor, followers) in enumerate(self.groups):
            every = sorted(followers) == [l for l in range(hs.L) if hs.anchor_of[l] == anchor]
            inline = bool(followers) and self.inline_shared and every
            if inline:
                f = self.flags | H.WITH_SHARED
                if through and self.fused:   # the shared layers' write-through before they are read
                    for fl in followers:
                        hs.writeback(fl, pos[fl:fl + 1], self.num_reqs, stream=self.compute,
                                     new_rows=new_rows[fl] if new_rows is not None else None)
            else:
                f = self.flags | (H.RECORD_PLAN if followers else 0)
            if self.resident is not None or self.sel_block_tokens > 1 or seq_lens is not None:
                fused = through and self.fused
                res = self.resident
                hs.resolve_ex(anchor, sel[gi], out[gi], self.num_reqs, newest,
                              pos[anchor] if fused else None,
                              new_rows[anchor] if (fused and new_rows is not None) else None,
                              res[0] if res is not None else None,
                              res[1] if res is not None else 0, self.sel_block_tokens, f,
                              stream=self.compute, seq_lens=seq_lens)
            elif through and self.fused:
                hs.resolve_step(anchor, sel[gi], out[gi], self.num_reqs, newest, pos[anchor],
                                new_rows[anchor] if new_rows is not None else None, f,
                                stream=self.compute)
            else:
                hs.resolve(anchor, sel[gi], out[gi], self.num_reqs, newest, f, stream=self.compute)
            if inline:
                for fi in range(len(followers)):
                    self.ev_follow[gi][fi].record(self.compute)
            elif followers:
                self.ev_anchor[gi].record(self.compute)
                self.side.wait_event(self.ev_anchor[gi])
                if self.group_replay and every:
                    if through and self.fused:   # the shared layers' own write-through first
                        for fl in followers:
                            hs.writeback(fl, pos[fl:fl + 1], self.num_reqs, stream=self.side,
                                         new_rows=new_rows[fl] if new_rows is not None else None)
                    hs.prefetch_plan(anchor, -1, self.num_reqs, stream=self.side)
                    for fi in range(len(followers)):
                        self.ev_follow[gi][fi].record(self.side)
                else:
                    for fi, fl in enumerate(followers):
                        if through and self.fused:   # the shared layer's own write-through first
                            hs.writeback(fl, pos[fl:fl + 1], self.num_reqs, stream=self.side,
                                         new_rows=new_rows[fl] if new_rows is not None else None)
                        hs.prefetch_plan(anchor, fl, self.num_reqs, stream=self.side)
                        self.ev_follow[gi][fi].record(self.side)
        # a shared layer's attention would wait on its own event; at the end of
        # the step the caller's stream waits for everything
        for gi, (_, followers) in enumerate(self.groups):
            for fi in range(len(followers)):
                cur.wait_event(self.ev_follow[gi][fi])
                self.compute.wait_event(self.ev_follow[gi][fi])
        self.ev_side_done.record(self.compute)
        cur.wait_event(self.ev_side_done)
