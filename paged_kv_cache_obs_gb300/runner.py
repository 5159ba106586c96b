"""Device-side plumbing around the C-ABI for one compression batch.

Builds the allocator state of a workload (reserved blocks, prefix-cache references), plans
the destination tables with zp_plan_compress, uploads tables and metadata, and launches
zp_compress.  No arithmetic of the method happens here.
"""
from __future__ import annotations

import numpy as np
import torch

from . import zipage


class CompressionBatch:
    def __init__(self, inp, device="cuda", pool=None):
        """inp: synth.Inputs (its tensors may live on the CPU or on `device`)."""
        self.inp = inp
        self.wl = wl = inp.wl
        self.params = wl.params()
        R = inp.num_compress
        NB = inp.pool.shape[1]
        self.alloc = zipage.zp_alloc_create(NB)
        used = np.nonzero(inp.refcount)[0].astype(np.int32)
        zipage.zp_alloc_reserve(self.alloc, used)
        extra = np.repeat(np.arange(NB, dtype=np.int32), np.maximum(inp.refcount - 1, 0))
        if len(extra):
            zipage.zp_incref(self.alloc, extra)
        self.tables = np.ascontiguousarray(inp.block_tables[:R])
        self.n_max_req = inp.n_max_req
        if self.n_max_req is None:
            self.dst_tables = zipage.zp_plan_compress(self.alloc, self.tables, wl.n_max)
        else:
            self.dst_tables = zipage.zp_plan_compress_budgets(self.alloc, self.tables, self.n_max_req)
        dev = torch.device(device)
        self.device = dev
        self.pool = pool if pool is not None else inp.pool.to(dev)
        self.d_tables = torch.from_numpy(self.tables).to(dev)
        self.d_dst = torch.from_numpy(self.dst_tables).to(dev)
        self.d_seq = torch.from_numpy(np.ascontiguousarray(inp.seq_len[:R])).to(dev)
        self.d_qslot = torch.from_numpy(inp.qslot).to(dev)
        self.obs_q = inp.obs_q.to(dev)
        self.gs = inp.global_scores.to(dev)
        # the row length of the global scores is the longest sequence the call may hold (more
        # than n_max*b only when requests left a long prefill)
        self.seq_len = np.ascontiguousarray(inp.seq_len[:R])
        row = inp.global_scores.shape[-1]
        self.max_seq_len = row if row != wl.L else 0
        self.workspace = zipage.new_workspace(
            zipage.zp_compress_workspace_size(self.params, R, self.max_seq_len), dev)
        self.d_nmax = None if self.n_max_req is None else torch.from_numpy(self.n_max_req).to(dev)
        self.debug = None

    def enable_debug(self):
        R, nl, Hkv = self.inp.num_compress, self.wl.num_layers, self.wl.num_kv_heads
        L = self.max_seq_len or self.wl.L
        z = lambda dt: torch.zeros((R, nl, Hkv, L), dtype=dt, device=self.device)
        self.debug = {"attn": z(torch.float32), "redund": z(torch.float32), "score": z(torch.float32),
                      "keep": z(torch.int32)}
        return self.debug

    def launch(self, stream=None, layers=None):
        """Queues the pass (over `layers` = (begin, count) only, when given)."""
        zipage.zp_compress(self.pool, self.d_tables, self.d_seq, self.d_qslot, self.d_dst, self.obs_q,
                           self.gs, self.params, self.workspace, debug=self.debug, stream=stream,
                           max_seq_len=self.max_seq_len, n_max_per_req=self.d_nmax, layers=layers)

    def error(self, stream=None) -> int:
        return zipage.zp_read_error(self.workspace, stream)

    def commit(self, stream=None):
        if self.n_max_req is None:
            zipage.zp_commit_compress(self.alloc, self.tables, self.dst_tables, self.wl.n_max, stream=stream,
                                      block_size=self.wl.block_size, seq_len=self.seq_len)
        else:
            zipage.zp_commit_compress_budgets(self.alloc, self.tables, self.dst_tables, self.n_max_req,
                                              self.wl.n_max, stream=stream, block_size=self.wl.block_size,
                                              seq_len=self.seq_len)

    def close(self):
        if self.alloc is not None:
            zipage.zp_alloc_destroy(self.alloc)
            self.alloc = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
