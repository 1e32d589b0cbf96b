"""Resident block tables for the three-tier resolve (input generation only).

In the vLLM design (docs.vllm.ai "HiSparse local KV offload architecture",
"Resident device pages" and "P/D import target") a request either lands whole
in resident device pages, when its prefix fits the device pools, or in the host
tier; pages of a host-tier request that are needed immediately are also
mirrored into resident pages.  These tables give that shape: the first
``full`` requests are resident over their whole context, and every other
request has the blocks covering its most recent ``window`` positions resident
(which includes the newest token).  Block indices are distinct across the
batch (request r's block b has index r * nblk + b), as a block table into one
shared store would have them.
"""
import numpy as np


def resident_tables(w, tokens_per_block=64, full=1, window=1024):
    """int32 [steps][R][nblk]: the resident block table before each decode step.

    ``nblk`` covers every host row (P positions).  Step t's context ends at
    position L_ctx + t (the newest token) for write-through workloads, else
    at L_ctx - 1.
    """
    tok = int(tokens_per_block)
    nblk = -(-w.P // tok)
    out = np.full((w.steps, w.R, nblk), -1, np.int32)
    ids = (np.arange(w.R, dtype=np.int64)[:, None] * nblk + np.arange(nblk)[None, :]).astype(np.int32)
    for t in range(w.steps):
        end = w.L_ctx + t if w.write_through else w.L_ctx - 1   # last valid position
        for r in range(w.R):
            if r < full:
                hi = end // tok + 1
                out[t, r, :hi] = ids[r, :hi]
            else:
                lo = max(0, end - window + 1) // tok
                hi = end // tok + 1
                out[t, r, lo:hi] = ids[r, lo:hi]
    return out
