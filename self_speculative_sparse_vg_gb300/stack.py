"""A multi-layer self-speculative decode loop around the three calls.

The attention stack of a decoder (by default Llama-3-8B-shaped: 32 layers,
hidden 4096, 32 query / 8 KV heads of 128) with random-initialised Q/K/V
projections.  Each iteration drafts k tokens with sparse attention over the
index sets chosen by the previous verification, verifies the k + 1 block with
full attention and Collect-2-Query capture, selects the next index sets per
layer, accepts a Bernoulli prefix of the drafts and commits accepted + 1
tokens (Vegas: Self-Speculative Decoding with Verification-Guided Sparse
Attention, "The pith", "Core claim" and Figure 1).

What stands in for the parts of a model outside the attention path:
  * layer input      h = bf16(x / sqrt(mean(x^2) + 1e-6))  (unit-gain RMS norm)
  * projections      q, k, v = bf16(h W_q), bf16(h W_k), bf16(h W_v), computed
                     in float64 so that the bf16 values do not depend on the
                     summation order
  * residual         x <- x + o   (no output projection, RoPE or MLP)
  * next token       the input vector of the token after position p is the
                     RMS-normalised final residual of position p (stands in
                     for LM head, sampling and embedding lookup)
  * acceptance       the accepted count of an iteration is the number of
                     leading ones of k Bernoulli(p) draws (stands in for
                     speculative sampling)

Positions: with n tokens in the cache, draft step t (1..k) processes the token
at position n + t - 1, writes its K/V there and attends the selection plus the
dense tail [tail_start, n + t).  The verify block holds positions n .. n + k;
its rows rewrite their K/V, attend causally and are captured at rows 0 and k;
the selection covers prefix [0, n).  After accepting a drafts the cache holds
n + a + 1 tokens, the next input comes from verify row a, and the next drafts'
tail starts at n.  A first one-row verify of the first token seeds the
selection.

The projections, norms and K/V writes are PyTorch plumbing; every attention
step runs in libvg's kernels through the C ABI.
"""
from __future__ import annotations

from typing import Callable, List, Optional

import torch

from . import vg
from .workloads import (PAGE_SIZE, StackSpec, make_acceptance, make_stack_context,
                        make_stack_embedding, make_stack_weights)

RMS_EPS = 1e-6


def accepted_counts(draws: torch.Tensor) -> torch.Tensor:
    """Leading ones along the last axis of a bool tensor."""
    return torch.cumprod(draws.to(torch.int64), dim=-1).sum(dim=-1)


def _rms(x: torch.Tensor) -> torch.Tensor:
    return x / torch.sqrt((x * x).mean(dim=-1, keepdim=True) + RMS_EPS)


class DecodeStack:
    """Device state of the stack (weights, paged K/V per layer, selections)
    and the decode loop.

    gen_device: where the seeded inputs are drawn (the values depend on it);
    they are then moved to `device`.  record(kind, layer, tensors), if given,
    is called after every attention call with kind "seed", "draft" or
    "verify" (tensors stay on the device).  force_selection(kind, layer), if
    given, is called once after each selection (after `record`); a returned
    (indices, counts) pair replaces the selection the next drafts use, so
    that two decode loops can be run on one sequence of selections.
    timing: if a list, every attention call appends (kind, start, end) CUDA
    events recorded around it on the current stream ("verify", "select",
    "draft")."""

    def __init__(self, spec: StackSpec, device="cuda", gen_device=None,
                 record: Optional[Callable] = None,
                 force_selection: Optional[Callable] = None):
        self.spec = s = spec
        self.device = dev = torch.device(device)
        gen_device = dev if gen_device is None else torch.device(gen_device)
        B, Hq, Hkv, d = s.batch, s.num_q_heads, s.num_kv_heads, s.head_dim
        self.R = s.n_drafts + 1
        self.nq, self.nk = Hq * d, Hkv * d
        self.w = []
        for l in range(s.layers):
            wq, wk, wv = make_stack_weights(s, l, gen_device)
            self.w.append(torch.cat([wq, wk, wv], dim=1).to(dev).double())
        # page table shared by the layers: sequence b owns a contiguous run of pages
        npages = [(L + s.room + self.R + PAGE_SIZE - 1) // PAGE_SIZE for L in s.prefix_lens]
        self.max_pages = max(npages)
        table = torch.full((B, self.max_pages), -1, dtype=torch.int32)
        self.first_page, off = [], 0
        for b, n in enumerate(npages):
            table[b, :n] = torch.arange(off, off + n, dtype=torch.int32)
            self.first_page.append(off)
            off += n
        self.num_pages = off
        self.page_table = table.to(dev)
        self.kp, self.vp = [], []
        for l in range(s.layers):
            kp = torch.zeros(off, Hkv, PAGE_SIZE, d, dtype=torch.bfloat16, device=dev)
            vp = torch.zeros_like(kp)
            ks, vs = make_stack_context(s, l, gen_device)
            for b, L in enumerate(s.prefix_lens):
                for src, pool in ((ks[b], kp), (vs[b], vp)):
                    src = src.to(dev)
                    full, rem, p0 = L // PAGE_SIZE, L % PAGE_SIZE, self.first_page[b]
                    pool[p0:p0 + full] = src[:, :full * PAGE_SIZE].reshape(
                        Hkv, full, PAGE_SIZE, d).permute(1, 0, 2, 3)
                    if rem:
                        pool[p0 + full, :, :rem] = src[:, full * PAGE_SIZE:]
            del ks, vs
            self.kp.append(kp)
            self.vp.append(vp)
        self.kv = [vg.PagedKV(self.kp[l], self.vp[l], self.page_table) for l in range(s.layers)]
        self.e = make_stack_embedding(s, gen_device).to(dev)      # input of the next token
        self.lens = torch.tensor(s.prefix_lens, dtype=torch.int32, device=dev)
        self.tail_start = self.lens.clone()
        self.rows = Hkv if s.per_head else 1
        self.cap = s.n_sel_max
        self.capture = torch.zeros(B, Hkv, s.max_prefix, dtype=torch.float32, device=dev)
        self.indices = [torch.full((B, self.rows, self.cap), -1, dtype=torch.int32, device=dev)
                        for _ in range(s.layers)]
        self.counts = [torch.zeros(B, self.rows, dtype=torch.int32, device=dev)
                       for _ in range(s.layers)]
        # cache slots of the selections (written by the selector); a forced
        # selection replaces the positions, so the drafts then translate them
        # through the page table instead
        self.slots = None if force_selection is not None else [
            torch.full((B, self.rows, self.cap), -1, dtype=torch.int32, device=dev)
            for _ in range(s.layers)]
        self.max_tail = 2 * s.n_drafts + 1
        self.ws_verify = {r: vg.zero_workspace(
            vg.verify_workspace_bytes(B, r, Hq, Hkv, d, s.max_prefix), dev) for r in (1, self.R)}
        self.ws_select = vg.zero_workspace(
            vg.select_workspace_bytes(B, Hkv, s.max_prefix, s.per_head), dev)
        self.ws_draft = vg.zero_workspace(
            vg.sparse_draft_workspace_bytes(B, Hq, Hkv, d, self.cap, self.max_tail), dev)
        self.flag = torch.zeros(1, dtype=torch.int32, device=dev)
        self.draws = make_acceptance(s)
        self.iteration = 0
        self.accepted: List[torch.Tensor] = []
        self.record = record
        self.force_selection = force_selection
        self.timing: Optional[list] = None

    # ------------------------------------------------------------ pieces
    def _qkv(self, l, x):
        """x float64 [..][hidden] -> bf16 q [..][Hq][d], k and v [..][Hkv][d]."""
        s = self.spec
        h = _rms(x).to(torch.bfloat16).double()
        y = (h @ self.w[l]).to(torch.bfloat16)
        shp = x.shape[:-1]
        q = y[..., :self.nq].reshape(*shp, s.num_q_heads, s.head_dim)
        k = y[..., self.nq:self.nq + self.nk].reshape(*shp, s.num_kv_heads, s.head_dim)
        v = y[..., self.nq + self.nk:].reshape(*shp, s.num_kv_heads, s.head_dim)
        return q.contiguous(), k, v

    def _write_kv(self, l, k, v, pos):
        """k, v [B][n][Hkv][d] to positions pos[b] + 0..n-1."""
        n = k.shape[1]
        p = pos[:, None].long() + torch.arange(n, device=self.device)[None, :]
        phys = torch.gather(self.page_table.long(), 1, p // PAGE_SIZE)
        slot = p % PAGE_SIZE
        self.kp[l][phys, :, slot] = k
        self.vp[l][phys, :, slot] = v

    def _timed(self, kind, fn, *args, **kw):
        if self.timing is None:
            return fn(*args, **kw)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        r = fn(*args, **kw)
        b.record()
        self.timing.append((kind, a, b))
        return r

    def _verify_select(self, l, q, R):
        s = self.spec
        out = torch.empty(s.batch, R, s.num_q_heads, s.head_dim, dtype=torch.bfloat16,
                          device=self.device)
        self._timed("verify", vg.verify_attention, self.kv[l], q, self.lens, s.max_prefix,
                    s.softmax_scale, out, vg.CAPTURE_GROUP_SUM, self.capture, 0,
                    self.ws_verify[R], self.flag)
        self._timed("select", vg.select_kv, self.capture, vg.CAPTURE_GROUP_SUM, self.lens,
                    s.num_q_heads, s.num_kv_heads, s.max_prefix, s.top_k, s.n_sink, s.n_recent,
                    s.per_head, self.indices[l], self.counts[l], self.flag,
                    workspace=self.ws_select, kv=self.kv[l],
                    slots=None if self.slots is None else self.slots[l])
        return out

    def _forced(self, kind, l):
        if self.force_selection is None:
            return
        r = self.force_selection(kind, l)
        if r is not None:
            self.indices[l].copy_(r[0])
            self.counts[l].copy_(r[1])

    def seed_selection(self):
        """A one-row verify of the first token over the initial context
        seeds every layer's selection; the token is committed."""
        s = self.spec
        x = self.e[:, None, :]                                   # [B][1][H]
        for l in range(s.layers):
            q, k, v = self._qkv(l, x)
            self._write_kv(l, k, v, self.lens)
            out = self._verify_select(l, q, 1)
            if self.record:
                self.record("seed", l, dict(out=out, capture=self.capture,
                                            indices=self.indices[l], counts=self.counts[l]))
            self._forced("seed", l)
            x = x + out.double().reshape(s.batch, 1, -1)
        self.tail_start = self.lens.clone()
        self.lens = self.lens + 1
        self.e = _rms(x[:, 0])

    def step(self):
        """One draft/verify iteration."""
        s = self.spec
        B, k = s.batch, s.n_drafts
        block = [self.e]                                         # inputs of positions n .. n+k
        for t in range(1, k + 1):
            pos = self.lens + (t - 1)
            cur = pos + 1
            x = block[-1]
            for l in range(s.layers):
                q, kk, vv = self._qkv(l, x)
                self._write_kv(l, kk[:, None], vv[:, None], pos)
                out = torch.empty(B, s.num_q_heads, s.head_dim, dtype=torch.bfloat16,
                                  device=self.device)
                self._timed("draft", vg.sparse_draft_attention, self.kv[l], q, self.indices[l],
                            self.counts[l], s.per_head, self.tail_start, cur, self.max_tail,
                            s.softmax_scale, out, self.ws_draft, self.flag,
                            slots=None if self.slots is None else self.slots[l])
                if self.record:
                    self.record("draft", l, dict(out=out, t=t))
                x = x + out.double().reshape(B, -1)
            block.append(_rms(x))
        X = torch.stack(block, dim=1)                            # [B][k+1][H]
        for l in range(s.layers):
            q, kk, vv = self._qkv(l, X)
            self._write_kv(l, kk, vv, self.lens)
            out = self._verify_select(l, q, k + 1)
            if self.record:
                self.record("verify", l, dict(out=out, capture=self.capture,
                                              indices=self.indices[l], counts=self.counts[l]))
            self._forced("verify", l)
            X = X + out.double().reshape(B, k + 1, -1)
        a = accepted_counts(self.draws[self.iteration])          # [B], host
        self.accepted.append(a)
        a_dev = a.to(self.device)
        self.tail_start = self.lens.clone()
        self.lens = self.lens + (a_dev + 1).to(torch.int32)
        self.e = _rms(X[torch.arange(B, device=self.device), a_dev])
        self.iteration += 1

    def launches_per_iteration(self) -> int:
        """Kernels per layer and draft/verify iteration: k drafts, the verify
        (+ split merge) and the selection."""
        s = self.spec
        merge = 1 if self.ws_verify[self.R].numel() > 1 else 0
        with torch.cuda.device(self.device):
            sel = vg.select_launches(vg.CAPTURE_GROUP_SUM, s.batch, s.num_kv_heads, s.max_prefix,
                                     s.per_head)
        return s.n_drafts + 1 + merge + sel

    def run(self, iterations: Optional[int] = None):
        self.seed_selection()
        n = self.spec.iterations if iterations is None else iterations
        for _ in range(n):
            self.step()
        return self
