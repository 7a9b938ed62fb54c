"""One decode step of one layer through the C ABI: verify (k+1 rows, capture)
-> select -> k sparse draft calls.  Holds the device buffers of a workload;
every computation happens in libvg's kernels."""
from __future__ import annotations

import ctypes
from dataclasses import dataclass, field
from typing import Optional

import torch

from . import vg
from .workloads import Inputs, WorkloadSpec


@dataclass
class DecodeStep:
    spec: WorkloadSpec
    device: torch.device
    kv: vg.PagedKV
    q_verify: torch.Tensor          # [B][R][Hq][d]
    draft_q: torch.Tensor           # [k][B][Hq][d]
    prefix_lens: torch.Tensor       # int32 [B]
    capture_mode: int
    per_head: bool
    capture: torch.Tensor
    out_verify: torch.Tensor
    indices: torch.Tensor
    counts: torch.Tensor
    out_draft: torch.Tensor         # [k][B][Hq][d]
    tail_start: torch.Tensor
    cur_len: torch.Tensor           # [k][B]
    ws_verify: torch.Tensor
    ws_draft: torch.Tensor
    ws_select: torch.Tensor
    error_flag: torch.Tensor
    num_splits: int = 0
    # cache slots written by the selector beside the indices (None: the draft
    # kernel translates positions through the page table itself)
    slots: Optional[torch.Tensor] = None
    extra: dict = field(default_factory=dict)
    # The step's inputs (q_verify, draft_q) and results (out_verify,
    # out_draft; indices, counts) are views into three flat buffers, so that a
    # host round trip of a step is one copy in and two copies out.
    io_in: Optional[torch.Tensor] = None      # bf16: q_verify, then draft_q
    io_out: Optional[torch.Tensor] = None     # bf16: out_verify, then out_draft
    io_sel: Optional[torch.Tensor] = None     # int32: indices, then counts

    @classmethod
    def create(cls, inp: Inputs, device="cuda", capture_mode=vg.CAPTURE_GROUP_SUM,
               per_head: Optional[bool] = None, num_splits=0, use_slots=True):
        s = inp.spec
        dev = torch.device(device)
        per_head = s.per_head if per_head is None else per_head
        B, R, Hq, Hkv, d = s.batch, s.n_rows, s.num_q_heads, s.num_kv_heads, s.head_dim
        Lmax = s.max_prefix
        kv = vg.PagedKV(inp.k_pages.to(dev), inp.v_pages.to(dev), inp.page_table.to(dev))
        if capture_mode == vg.CAPTURE_ROWS:
            capture = torch.zeros(B, Hq, 2, Lmax, dtype=torch.float32, device=dev)
        elif capture_mode == vg.CAPTURE_ALL_ROWS:
            capture = torch.zeros(vg.all_rows_capture_floats(B, Hq, R, Lmax), dtype=torch.float32,
                                  device=dev)
        else:
            capture = torch.zeros(B, Hkv, Lmax, dtype=torch.float32, device=dev)
        rows = Hkv if per_head else 1
        cap = min(Lmax, s.n_sel_max)
        prefix = torch.tensor(s.prefix_lens, dtype=torch.int32, device=dev)
        k = s.n_drafts
        cur = torch.stack([prefix + t for t in range(1, k + 1)]) if k else prefix[None][:0]
        wsv = vg.zero_workspace(vg.verify_workspace_bytes(B, R, Hq, Hkv, d, Lmax, num_splits), dev)
        wsd = vg.zero_workspace(vg.sparse_draft_workspace_bytes(B, Hq, Hkv, d, cap, max(k, 1)), dev)
        wss = vg.zero_workspace(vg.select_workspace_bytes(B, Hkv, Lmax, per_head), dev)
        nv, nd = B * R * Hq * d, max(k, 1) * B * Hq * d
        io_in = torch.zeros(nv + nd, dtype=torch.bfloat16, device=dev)
        q_verify = io_in[:nv].view(B, R, Hq, d)
        draft_q = io_in[nv:].view(max(k, 1), B, Hq, d)
        q_verify.copy_(inp.q_verify)
        draft_q[:k].copy_(inp.draft_q)
        io_out = torch.zeros(nv + nd, dtype=torch.bfloat16, device=dev)
        ni = B * rows * cap
        io_sel = torch.zeros(ni + B * rows, dtype=torch.int32, device=dev)
        indices = io_sel[:ni].view(B, rows, cap)
        indices.fill_(-7)
        slots = torch.full((B, rows, cap), -7, dtype=torch.int32, device=dev) if use_slots else None
        return cls(spec=s, device=dev, kv=kv, q_verify=q_verify, draft_q=draft_q[:k] if k else draft_q[:0],
                   prefix_lens=prefix, capture_mode=capture_mode, per_head=per_head,
                   capture=capture, out_verify=io_out[:nv].view(B, R, Hq, d),
                   indices=indices, counts=io_sel[ni:].view(B, rows),
                   out_draft=io_out[nv:].view(max(k, 1), B, Hq, d),
                   tail_start=prefix.clone(), cur_len=cur.contiguous(), ws_verify=wsv,
                   ws_draft=wsd, ws_select=wss, error_flag=torch.zeros(1, dtype=torch.int32, device=dev),
                   num_splits=num_splits, slots=slots, io_in=io_in, io_out=io_out, io_sel=io_sel)

    @property
    def max_tail(self):
        return max(self.spec.n_drafts, 1)

    # The C calls are made with argument tuples built once per stream (the
    # buffers never move), so a launch costs one ctypes call.
    def _args(self, kind, t, stream):
        s = torch.cuda.current_stream(self.device) if stream is None else stream
        key = (kind, t, s.cuda_stream)
        cache = self.extra.setdefault("args", {})
        if key in cache:
            return cache[key]
        p = lambda x: ctypes.c_void_p(x.data_ptr())  # noqa: E731
        sp, st = self.spec, ctypes.c_void_p(s.cuda_stream)
        kvs = self.extra.setdefault("kv_struct", self.kv.struct())
        B, R, Hq, d = self.q_verify.shape
        slots = None if self.slots is None else p(self.slots)
        kv_arg = None if self.slots is None else ctypes.byref(kvs)
        if kind == "verify":
            a = (ctypes.byref(kvs), p(self.q_verify), p(self.prefix_lens), B, R, Hq,
                 sp.max_prefix, ctypes.c_float(sp.softmax_scale), p(self.out_verify),
                 self.capture_mode, p(self.capture), self.num_splits, p(self.ws_verify),
                 self.ws_verify.numel(), p(self.error_flag), st)
        elif kind == "select" and self.capture_mode == vg.CAPTURE_ALL_ROWS:
            a = (p(self.capture), R, p(self.prefix_lens), B, Hq, sp.num_kv_heads,
                 sp.max_prefix, sp.top_k, sp.n_sink, sp.n_recent, int(self.per_head),
                 p(self.indices), p(self.counts), self.indices.shape[-1], kv_arg, slots,
                 p(self.ws_select), self.ws_select.numel(), p(self.error_flag), st)
        elif kind == "select":
            a = (p(self.capture), self.capture_mode, p(self.prefix_lens), B, Hq, sp.num_kv_heads,
                 sp.max_prefix, sp.top_k, sp.n_sink, sp.n_recent, int(self.per_head),
                 p(self.indices), p(self.counts), self.indices.shape[-1], kv_arg, slots,
                 p(self.ws_select), self.ws_select.numel(), p(self.error_flag), st)
        else:
            a = (ctypes.byref(kvs), p(self.draft_q[t - 1]), p(self.indices), slots, p(self.counts),
                 int(self.per_head), self.indices.shape[-1], p(self.tail_start),
                 p(self.cur_len[t - 1]), B, Hq, self.max_tail, ctypes.c_float(sp.softmax_scale),
                 p(self.out_draft[t - 1]), p(self.ws_draft), self.ws_draft.numel(),
                 p(self.error_flag), st)
        cache[key] = a
        return a

    def verify(self, stream=None):
        vg._check("vg_verify_attention", vg._lib.vg_verify_attention(*self._args("verify", 0, stream)))

    def select(self, stream=None):
        if self.capture_mode == vg.CAPTURE_ALL_ROWS:
            vg._check("vg_select_kv_weights",
                      vg._lib.vg_select_kv_weights(*self._args("select", 0, stream)))
        else:
            vg._check("vg_select_kv", vg._lib.vg_select_kv(*self._args("select", 0, stream)))

    def draft(self, t: int, stream=None):
        """Draft step t = 1..k: query at position L + t - 1, tail [L, L + t)."""
        vg._check("vg_sparse_draft_attention",
                  vg._lib.vg_sparse_draft_attention(*self._args("draft", t, stream)))

    def run(self, stream=None):
        self.verify(stream)
        self.select(stream)
        for t in range(1, self.spec.n_drafts + 1):
            self.draft(t, stream)

    def launches_per_step(self) -> int:
        """Kernels of one step: verify (+ its split merge when it has more
        than one split), the selection's kernels, one kernel per draft step."""
        merge = 1 if self.ws_verify.numel() > 1 else 0
        sp = self.spec
        with torch.cuda.device(self.device):
            sel = vg.select_launches(self.capture_mode, sp.batch, sp.num_kv_heads, sp.max_prefix,
                                     self.per_head)
        return 1 + merge + sel + sp.n_drafts
