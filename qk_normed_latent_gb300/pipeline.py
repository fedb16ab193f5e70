"""Run the decode path (absorb -> append -> decode) on a synthetic workload.

Device-side driver used by the tests, the benchmark and the smoke check.  It
only moves the seeded inputs of `workloads` to the GPU and calls the library;
all arithmetic happens in the CUDA kernels.
"""
from __future__ import annotations

import numpy as np
import torch

import workloads as W

from . import (F32, BF16, append, decode_workspace_size, decode_raw, make_decode_args, prepare_absorb_query,
               prepare_append)

_TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
# quiet-NaN bit patterns written into untouched cache slots
SENTINEL_BF16 = 0x7FC1
SENTINEL_F32 = 0x7FC00001
SENTINEL_F16 = 0x7E01


def packed(parts, device, empty=False):
    """One device byte buffer holding the given arrays back to back (each part
    256-byte aligned); returns the buffer and a tensor view of each part.  A step's
    inputs (or outputs) then cross PCIe / C2C in a single copy.  With `empty` the
    parts are (shape, dtype) pairs and the buffer is left unfilled."""
    metas = []
    off = 0
    for part in parts:
        if empty:
            shape, dt = part
            nbytes = int(np.prod(shape)) * torch.tensor([], dtype=dt).element_size()
        else:
            arr = np.ascontiguousarray(part)
            shape, dt, nbytes = arr.shape, torch.from_numpy(arr[:0].copy()).dtype, arr.nbytes
        off = (off + 255) & ~255
        metas.append((off, shape, dt, nbytes, None if empty else arr))
        off += nbytes
    buf = torch.empty(max(off, 1), dtype=torch.uint8, device=device)
    views = []
    for o, shape, dt, nbytes, arr in metas:
        v = buf[o:o + nbytes].view(dt).view(shape)
        if arr is not None:
            v.copy_(torch.from_numpy(arr))
        views.append(v)
    return buf, views


def sentinel_fill(t: torch.Tensor) -> None:
    if t.dtype == torch.bfloat16:
        t.view(torch.int16).fill_(SENTINEL_BF16)
    elif t.dtype == torch.float16:
        t.view(torch.int16).fill_(SENTINEL_F16)
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
        self.ak = torch.empty((self.num_slots, w.G), dtype=_TORCH_DT[w.alpha_dtype], device=d)
        if sentinel:
            sentinel_fill(self.kv)
            sentinel_fill(self.ak)
        self.seq_lens = torch.from_numpy(self.lens.astype(np.int32)).to(d)
        self.page_table = torch.from_numpy(table).to(d) if self.paged else None
        q, qr = W.queries(w)
        self.q_tilde = torch.empty((w.B, w.s_q, w.H, w.d_c), dtype=cdt, device=d)
        self.alpha_q = torch.empty((w.B, w.s_q, w.H), dtype=torch.float32, device=d)
        # the step's results, o and lse, in one buffer
        self.step_out, (self.o, self.lse) = packed(
            [((w.B, w.s_q, w.H, w.d_c), o_dtype), ((w.B, w.s_q, w.H), torch.float32)], d, empty=True)
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
        # the step's inputs -- queries, RoPE queries and the new tokens -- in one buffer
        parts = [q.reshape(w.rows, w.H, w.d_h), qr]
        if n_new:
            parts += [np.concatenate(new_c), np.concatenate(new_r), np.concatenate(new_slots).astype(np.int64)]
        self.step_in, views = packed(parts, d)
        self.q, self.q_rope = views[0], views[1]
        if n_new:
            self.c_new, self.r_new, self.slots_new = views[2], views[3], views[4]
        else:
            self.c_new = self.r_new = self.slots_new = None
        self.workspace = None
        self.args = None
        self._absorb = self._append = None

    # -- the three calls -------------------------------------------------------
    def absorb(self, stream=None):
        w = self.w
        if self._absorb is None:             # the tensors never move: marshal once
            self._absorb = prepare_absorb_query(self.q, self.gq, self.gk, self.wk, w.eps,
                                                self.q_tilde.view(w.rows, w.H, w.d_c),
                                                self.alpha_q.view(w.rows, w.H), plain=self.plain)
        self._absorb(stream)

    def append_step(self, stream=None):
        if self.c_new is None:
            return
        if self._append is None:
            self._append = prepare_append(self.c_new, self.r_new, self.wk, self.grk, self.slots_new, self.kv,
                                          self.ak, self.w.eps, plain=self.plain)
        self._append(stream)

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
