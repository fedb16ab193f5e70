"""Run the decode path (absorb -> append -> decode) on a synthetic workload.

Device-side driver used by the tests, the benchmark and the smoke check.  It
only moves the seeded inputs of `workloads` to the GPU and calls the library;
all arithmetic happens in the CUDA kernels.
"""
from __future__ import annotations

import numpy as np
import torch

import workloads as W

from . import (F32, BF16, absorb_query, append, decode_workspace_size, decode_raw, make_decode_args)

_TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16}
# quiet-NaN bit patterns written into untouched cache slots
SENTINEL_BF16 = 0x7FC1
SENTINEL_F32 = 0x7FC00001


def sentinel_fill(t: torch.Tensor) -> None:
    if t.dtype == torch.bfloat16:
        t.view(torch.int16).fill_(SENTINEL_BF16)
    elif t.dtype == torch.float32:
        t.view(torch.int32).fill_(SENTINEL_F32)
    else:
        raise ValueError(t.dtype)


class DeviceState:
    """Device tensors of one workload.  Prefill writes every token except the
    last `n_append` of each sequence; `step()` appends those and decodes."""

    def __init__(self, w: W.Workload, plain: bool = False, o_dtype=torch.float32, device: str = "cuda",
                 prefill_chunk: int = 1 << 18, sentinel: bool = True, keep_host: bool = False):
        self.w = w
        self.plain = plain
        self.dev = torch.device(device)
        self.lens = W.seq_lens(w)
        self.page_size, self.max_pages, self.num_slots, table = W.page_layout(w, self.lens)
        self.table_np = table
        self.paged = w.page_size is not None
        wk, gq, gk, grq, grk = W.weights(w)
        d = self.dev
        self.wk = torch.from_numpy(wk).to(d)
        self.gq = torch.from_numpy(gq).to(d)
        self.gk = torch.from_numpy(gk).to(d)
        self.grq = torch.from_numpy(grq).to(d)
        self.grk = torch.from_numpy(grk).to(d)
        cdt = _TORCH_DT[w.cache_dtype]
        self.kv = torch.empty((self.num_slots, w.d_c + w.d_r), dtype=cdt, device=d)
        self.ak = torch.empty((self.num_slots, w.G), dtype=torch.float32, device=d)
        if sentinel:
            sentinel_fill(self.kv)
            sentinel_fill(self.ak)
        self.seq_lens = torch.from_numpy(self.lens.astype(np.int32)).to(d)
        self.page_table = torch.from_numpy(table).to(d) if self.paged else None
        q, qr = W.queries(w)
        self.q_host, self.qr_host = q, qr
        self.q = torch.from_numpy(q.reshape(w.rows, w.H, w.d_h)).to(d)
        self.q_rope = torch.from_numpy(qr).to(d)
        self.q_tilde = torch.empty((w.B, w.s_q, w.H, w.d_c), dtype=cdt, device=d)
        self.alpha_q = torch.empty((w.B, w.s_q, w.H), dtype=torch.float32, device=d)
        self.o = torch.empty((w.B, w.s_q, w.H, w.d_c), dtype=o_dtype, device=d)
        self.lse = torch.empty((w.B, w.s_q, w.H), dtype=torch.float32, device=d)
        # prefill, keeping the step's new tokens aside
        n_new = w.n_append
        new_c, new_r, new_slots = [], [], []
        self.host_seqs = [] if keep_host else None
        for b in range(w.B):
            c, r = W.sequence(w, b)
            L = c.shape[0]
            if keep_host:
                self.host_seqs.append((c, r))
            pre = L - n_new
            for s0 in range(0, pre, prefill_chunk):
                s1 = min(pre, s0 + prefill_chunk)
                slots = torch.from_numpy(W.slots_of(table, self.page_size, b, np.arange(s0, s1))).to(d)
                append(torch.from_numpy(c[s0:s1]).to(d), torch.from_numpy(r[s0:s1]).to(d), self.wk, self.grk,
                       slots, self.kv, self.ak, w.eps, plain=plain)
            if n_new:
                new_c.append(c[pre:])
                new_r.append(r[pre:])
                new_slots.append(W.slots_of(table, self.page_size, b, np.arange(pre, L)))
        if n_new:
            self.c_new = torch.from_numpy(np.concatenate(new_c)).to(d)
            self.r_new = torch.from_numpy(np.concatenate(new_r)).to(d)
            self.slots_new = torch.from_numpy(np.concatenate(new_slots)).to(d)
        else:
            self.c_new = self.r_new = self.slots_new = None
        self.workspace = None
        self.args = None

    # -- the three calls -------------------------------------------------------
    def absorb(self, stream=None):
        w = self.w
        absorb_query(self.q, self.gq, self.gk, self.wk, w.eps, self.q_tilde.view(w.rows, w.H, w.d_c),
                     self.alpha_q.view(w.rows, w.H), plain=self.plain, stream=stream)

    def append_step(self, stream=None):
        if self.c_new is not None:
            append(self.c_new, self.r_new, self.wk, self.grk, self.slots_new, self.kv, self.ak, self.w.eps,
                   plain=self.plain, stream=stream)

    def decode_args(self, num_splits: int = 0, force_simt: bool = False):
        w = self.w
        a = make_decode_args(self.q_tilde, self.alpha_q, self.q_rope, self.grq, self.kv, self.ak, self.seq_lens,
                             self.page_table, self.page_size, self.max_pages, w.G, w.scale, w.eps, self.o,
                             self.lse, plain=self.plain, force_simt=force_simt, num_splits=num_splits)
        need = decode_workspace_size(a)
        if need:
            if self.workspace is None or self.workspace.numel() < need:
                self.workspace = torch.empty(need, dtype=torch.uint8, device=self.dev)
            a.workspace, a.workspace_bytes = self.workspace.data_ptr(), self.workspace.numel()
        return a

    def decode(self, num_splits: int = 0, force_simt: bool = False, stream=None):
        self.args = self.decode_args(num_splits, force_simt)
        decode_raw(self.args, stream)

    def step(self, num_splits: int = 0, force_simt: bool = False, stream=None):
        """One pass of the whole path: absorb, append this step's tokens, decode."""
        self.absorb(stream)
        self.append_step(stream)
        if self.args is None or num_splits != self.args.num_splits:
            self.args = self.decode_args(num_splits, force_simt)
        decode_raw(self.args, stream)
