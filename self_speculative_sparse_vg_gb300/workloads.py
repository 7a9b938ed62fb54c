"""Seeded synthetic inputs for the verify / select / sparse-draft path.

This module only draws random numbers and lays them out (dense logical
layout for checking, paged layout for the kernels).  It holds none of the
attention or selection arithmetic, so both the float64 oracle and the CUDA
path can be fed from it without sharing any of the method's code.

Shapes follow the workloads the method is evaluated on: GQA decoder layers
shaped like Llama-3-8B (32 query / 8 KV heads, head_dim 128) and Qwen-14B
(40 / 8, head_dim 128), contexts of 2K to 128K tokens, k = 4..7 drafts, and a
selection budget of top-k plus sink and recent windows (Vegas: Self-Speculative
Decoding with Verification-Guided Sparse Attention, "Core claim" and the
Appendix B sparse-ratio discussion; A Sparse Glimpse of the Whole, "What
carries the argument").  No dataset is read: the long-context benchmarks the
pages measure on are stood in for by these seeded tensors.

Heavy hitters: a few prefix keys are pushed toward the mean direction of the
group's verify queries so that a correct top-k must recover them.  This is an
input construction, not part of the method.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import List, Optional

import torch

PAGE_SIZE = 16


@dataclass(frozen=True)
class WorkloadSpec:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    prefix_lens: tuple            # committed prefix length L_b per sequence
    n_drafts: int                 # k; the verify block has k+1 rows
    top_k: int
    n_sink: int
    n_recent: int
    seed: int
    heavy_frac: float = 0.0       # fraction of candidate positions boosted
    n_planted: int = 0            # exact count (overrides heavy_frac when > 0)
    planted_mode: str = "add"     # "add": K += s*sqrt(d)*u ; "replace": K = s*sqrt(d)*u
    planted_scale: float = 3.0
    shuffle_pages: bool = False
    extra_pages: int = 0          # spare physical pages (never referenced)
    per_head: bool = False

    @property
    def n_rows(self) -> int:
        return self.n_drafts + 1

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def max_prefix(self) -> int:
        return max(self.prefix_lens)

    @property
    def n_sel_max(self) -> int:
        return self.n_sink + self.n_recent + self.top_k


def _drawn_lengths(n: int, lo: int, hi: int, seed: int) -> tuple:
    g = torch.Generator().manual_seed(seed)
    return tuple(int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g))


# Named workloads.  Sizes are those of the evaluation the method targets.
WORKLOADS = {
    # Single layer, batch 1: 8 q heads / 2 kv heads, head_dim 64, 2K context,
    # 16 planted keys equal to 4x the query direction; k=4; 128 + 4 + 32.
    "tiny_d64_2k": WorkloadSpec(
        name="tiny_d64_2k", batch=1, num_q_heads=8, num_kv_heads=2, head_dim=64,
        prefix_lens=(2048,), n_drafts=4, top_k=128, n_sink=4, n_recent=32, seed=1,
        n_planted=16, planted_mode="replace", planted_scale=4.0),
    # Llama-3-8B-shaped layer, batch 1, 32K context, 1% heavy hitters; k=5;
    # 2048 + 4 + 64.
    "llama8b_32k": WorkloadSpec(
        name="llama8b_32k", batch=1, num_q_heads=32, num_kv_heads=8, head_dim=128,
        prefix_lens=(32768,), n_drafts=5, top_k=2048, n_sink=4, n_recent=64, seed=2,
        heavy_frac=0.01),
    # Same layer, batch 8, per-sequence context uniform in [16K, 64K], randomly
    # permuted page table; both selection modes are exercised.
    "llama8b_b8_16k_64k": WorkloadSpec(
        name="llama8b_b8_16k_64k", batch=8, num_q_heads=32, num_kv_heads=8, head_dim=128,
        prefix_lens=_drawn_lengths(8, 16384, 65536, 3), n_drafts=5, top_k=2048,
        n_sink=4, n_recent=64, seed=3, heavy_frac=0.01, shuffle_pages=True),
    # Qwen-14B-shaped layer, batch 1, 128K context, 0.5% heavy hitters; k=7;
    # 4096 + 4 + 128.
    "qwen14b_128k": WorkloadSpec(
        name="qwen14b_128k", batch=1, num_q_heads=40, num_kv_heads=8, head_dim=128,
        prefix_lens=(131072,), n_drafts=7, top_k=4096, n_sink=4, n_recent=128, seed=4,
        heavy_frac=0.005),
}


def small_spec(**kw) -> WorkloadSpec:
    """A small workload for quick parity cases (several tiles, ragged tail)."""
    base = WorkloadSpec(name="small", batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128,
                        prefix_lens=(1000, 517), n_drafts=3, top_k=64, n_sink=4,
                        n_recent=16, seed=11, heavy_frac=0.01)
    return replace(base, **kw)


@dataclass
class Inputs:
    spec: WorkloadSpec
    q_verify: torch.Tensor              # bf16 [B][R][Hq][d]
    k_dense: List[torch.Tensor]         # per b: bf16 [Hkv][n_b][d], n_b = L_b + R
    v_dense: List[torch.Tensor]
    draft_q: torch.Tensor               # bf16 [k][B][Hq][d]
    planted: List[torch.Tensor]         # per b: int64 planted positions
    page_table: torch.Tensor            # int32 [B][max_pages], -1 = unused
    k_pages: torch.Tensor               # bf16 [P][Hkv][16][d]
    v_pages: torch.Tensor
    extra: dict = field(default_factory=dict)

    @property
    def prefix_lens(self) -> torch.Tensor:
        return torch.tensor(self.spec.prefix_lens, dtype=torch.int32)


def _unit(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm()


def make_inputs(spec: WorkloadSpec, cache_extra: int = 0) -> Inputs:
    """Draw all inputs of `spec` on the CPU from its seed.

    cache_extra: additional cache positions per sequence beyond L_b + R
    (zero-filled K/V, used by tests that append tokens)."""
    s = spec
    B, R, Hq, Hkv, d, g = s.batch, s.n_rows, s.num_q_heads, s.num_kv_heads, s.head_dim, s.group
    assert Hq % Hkv == 0 and len(s.prefix_lens) == B
    gen = torch.Generator().manual_seed(s.seed)
    q_verify = torch.randn(B, R, Hq, d, generator=gen).to(torch.bfloat16)
    k_dense, v_dense, planted = [], [], []
    for b in range(B):
        L = s.prefix_lens[b]
        n = L + R
        k = torch.randn(Hkv, n + cache_extra, d, generator=gen)
        v = torch.randn(Hkv, n + cache_extra, d, generator=gen)
        if cache_extra:
            k[:, n:] = 0
            v[:, n:] = 0
        lo, hi = s.n_sink, max(s.n_sink, L - s.n_recent)
        n_cand = hi - lo
        n_pl = s.n_planted if s.n_planted > 0 else int(round(s.heavy_frac * L))
        n_pl = min(n_pl, n_cand)
        pos = (torch.randperm(n_cand, generator=gen)[:n_pl] + lo).sort().values
        if n_pl:
            qd = q_verify[b].double()                       # [R][Hq][d]
            for h in range(Hkv):
                u = _unit(qd[:, h * g:(h + 1) * g, :].sum(dim=(0, 1))).float()
                amp = s.planted_scale * math.sqrt(d)
                if s.planted_mode == "replace":
                    k[h, pos] = amp * u
                else:
                    k[h, pos] += amp * u
        k_dense.append(k.to(torch.bfloat16))
        v_dense.append(v.to(torch.bfloat16))
        planted.append(pos)
    draft_q = torch.randn(s.n_drafts, B, Hq, d, generator=gen).to(torch.bfloat16)
    page_table, k_pages, v_pages = to_paged(k_dense, v_dense, shuffle=s.shuffle_pages,
                                            seed=s.seed + 1000, extra_pages=s.extra_pages)
    return Inputs(spec=s, q_verify=q_verify, k_dense=k_dense, v_dense=v_dense, draft_q=draft_q,
                  planted=planted, page_table=page_table, k_pages=k_pages, v_pages=v_pages)


def to_paged(k_dense, v_dense, shuffle=False, seed=0, extra_pages=0, max_pages=None):
    """Lay dense per-sequence K/V ([Hkv][n_b][d]) into a page pool
    [P][Hkv][16][d] plus a page table [B][max_pages] (logical -> physical,
    -1 where unused).  Positions past n_b inside the last page are zero."""
    B = len(k_dense)
    Hkv, _, d = k_dense[0].shape
    npages = [(k.shape[1] + PAGE_SIZE - 1) // PAGE_SIZE for k in k_dense]
    total = sum(npages) + extra_pages
    mp = max(npages) if max_pages is None else max_pages
    if shuffle:
        phys = torch.randperm(total, generator=torch.Generator().manual_seed(seed))
    else:
        phys = torch.arange(total)
    kp = torch.zeros(total, Hkv, PAGE_SIZE, d, dtype=k_dense[0].dtype)
    vp = torch.zeros_like(kp)
    table = torch.full((B, mp), -1, dtype=torch.int32)
    off = 0
    for b in range(B):
        n = k_dense[b].shape[1]
        np_b = npages[b]
        ids = phys[off:off + np_b]
        off += np_b
        table[b, :np_b] = ids.to(torch.int32)
        for src, dst in ((k_dense[b], kp), (v_dense[b], vp)):
            pad = torch.zeros(Hkv, np_b * PAGE_SIZE, d, dtype=src.dtype)
            pad[:, :n] = src
            dst[ids] = pad.view(Hkv, np_b, PAGE_SIZE, d).permute(1, 0, 2, 3)
    return table, kp, vp


def make_capture(spec: WorkloadSpec, capture_mode: int, seed: int) -> torch.Tensor:
    """Synthetic captured logits for exercising a selector on its own (the
    same tensor is given to the kernel and to the checker).  Values are
    N(0, 3) rounded to multiples of 1/8, so exact ties are frequent, with a
    few large planted values.  capture_mode 1: [B][Hkv][Lmax];
    2: [B][Hq][2][Lmax] (float32)."""
    g = torch.Generator().manual_seed(seed)
    B, Hq, Hkv, Lmax = spec.batch, spec.num_q_heads, spec.num_kv_heads, spec.max_prefix
    shape = (B, Hkv, Lmax) if capture_mode == 1 else (B, Hq, 2, Lmax)
    x = torch.round(torch.randn(shape, generator=g) * 3.0 * 8.0) / 8.0
    flat = x.view(-1)
    hot = torch.randint(0, flat.numel(), (max(1, flat.numel() // 500),), generator=g)
    flat[hot] = 40.0
    return x.float()


def make_selection(spec: WorkloadSpec, per_head: bool, seed: int):
    """Synthetic index lists for exercising the sparse draft kernel on its
    own: per (sequence, row) a sorted set of min(L_b, budget) distinct prefix
    positions drawn uniformly, padded with -1.  Returns (indices int32
    [B][rows][cap], counts int32 [B][rows])."""
    g = torch.Generator().manual_seed(seed)
    B = spec.batch
    rows = spec.num_kv_heads if per_head else 1
    cap = min(spec.max_prefix, spec.n_sel_max)
    idx = torch.full((B, rows, cap), -1, dtype=torch.int32)
    cnt = torch.zeros(B, rows, dtype=torch.int32)
    for b, L in enumerate(spec.prefix_lens):
        n = min(L, spec.n_sel_max)
        for r in range(rows):
            pos = torch.randperm(L, generator=g)[:n].sort().values
            idx[b, r, :n] = pos.to(torch.int32)
            cnt[b, r] = n
    return idx, cnt


# ------------------------------------------------------------------ layer stack
@dataclass(frozen=True)
class StackSpec:
    """A decoder attention stack driven through several draft/verify
    iterations.  The Llama-3-8B-shaped default is 32 layers of hidden 4096,
    32 query / 8 KV heads of 128, batch 4 at contexts 32K/64K/96K/128K, k = 5
    drafts, a 2048 + 4 + 64 selection budget, 200 iterations and Bernoulli(0.7)
    acceptance of each draft."""
    name: str = "llama8b_stack32_b4"
    layers: int = 32
    hidden: int = 4096
    num_q_heads: int = 32
    num_kv_heads: int = 8
    head_dim: int = 128
    prefix_lens: tuple = (32768, 65536, 98304, 131072)
    n_drafts: int = 5
    top_k: int = 2048
    n_sink: int = 4
    n_recent: int = 64
    iterations: int = 200
    accept_p: float = 0.7
    per_head: bool = False
    seed: int = 6

    @property
    def batch(self) -> int:
        return len(self.prefix_lens)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def room(self) -> int:
        """Cache positions written past L_b over a run: the first token, then
        at most k + 1 committed per iteration, plus one block of k + 1 beyond."""
        return 1 + (self.iterations + 1) * (self.n_drafts + 1)

    @property
    def max_prefix(self) -> int:
        return max(self.prefix_lens) + self.room

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def n_sel_max(self) -> int:
        return self.n_sink + self.n_recent + self.top_k


STACKS = {"llama8b_stack32_b4": StackSpec()}


def small_stack(**kw) -> StackSpec:
    """A stack the float64 oracle runs in seconds: two layers, two sequences
    of a few thousand positions, a few iterations, the Llama-3-8B head shape."""
    base = StackSpec(name="small_stack", layers=2, prefix_lens=(1203, 2170), n_drafts=5,
                     top_k=96, n_sink=4, n_recent=32, iterations=4, seed=21)
    return replace(base, **kw)


def _gen(device, seed: int) -> torch.Generator:
    return torch.Generator(device=torch.device(device)).manual_seed(seed)


def make_stack_weights(spec: StackSpec, layer: int, device="cpu"):
    """Q, K, V projection weights of one layer: bf16 [hidden][heads * d],
    entries N(0, 1/hidden) (random initialisation; no checkpoint is read)."""
    s = spec
    g = _gen(device, s.seed * 7919 + 2 * layer)
    std = 1.0 / math.sqrt(s.hidden)
    out = []
    for n in (s.num_q_heads, s.num_kv_heads, s.num_kv_heads):
        w = torch.randn(s.hidden, n * s.head_dim, generator=g, device=device) * std
        out.append(w.to(torch.bfloat16))
    return tuple(out)


def make_stack_context(spec: StackSpec, layer: int, device="cpu"):
    """The initial context of one layer: per sequence b, bf16 K and V
    [Hkv][L_b][d] with entries N(0, 1)."""
    s = spec
    g = _gen(device, s.seed * 7919 + 2 * layer + 1)
    ks, vs = [], []
    for L in s.prefix_lens:
        ks.append(torch.randn(s.num_kv_heads, L, s.head_dim, generator=g, device=device)
                  .to(torch.bfloat16))
        vs.append(torch.randn(s.num_kv_heads, L, s.head_dim, generator=g, device=device)
                  .to(torch.bfloat16))
    return ks, vs


def make_stack_embedding(spec: StackSpec, device="cpu") -> torch.Tensor:
    """Input vector of the first decoded token of each sequence: float64
    [B][hidden], entries N(0, 1)."""
    g = _gen(device, spec.seed * 7919 - 1)
    return torch.randn(spec.batch, spec.hidden, generator=g, device=device, dtype=torch.float64)


def make_acceptance(spec: StackSpec) -> torch.Tensor:
    """Per iteration, sequence and draft a Bernoulli(accept_p) draw: bool
    [iterations][B][k].  These stand in for the accept/reject decisions of
    speculative sampling, which need a trained model."""
    g = torch.Generator().manual_seed(spec.seed * 7919 - 2)
    return torch.rand(spec.iterations, spec.batch, spec.n_drafts, generator=g) < spec.accept_p


def make_block_selection(spec: WorkloadSpec, frac: float, seed: int, overlap: float = 0.75):
    """Per verify row, a seeded set of 16-position prefix blocks for sparse
    verification: a core shared by all rows of the sequence (a share
    `overlap` of each row's blocks) plus row-private blocks, so adjacent rows
    overlap the way speculative rows do.  frac is the fraction of the
    sequence's prefix blocks a row selects (0 selects none, 1 all).
    Returns (blocks int32 [B][R][max_blocks] padded with -1, counts int32 [B][R])."""
    g = torch.Generator().manual_seed(seed)
    B, R = spec.batch, spec.n_rows
    nbl = [(L + PAGE_SIZE - 1) // PAGE_SIZE for L in spec.prefix_lens]
    want = [min(n, int(round(frac * n))) for n in nbl]
    max_blocks = max(1, max(want))
    blocks = torch.full((B, R, max_blocks), -1, dtype=torch.int32)
    counts = torch.zeros(B, R, dtype=torch.int32)
    for b, n in enumerate(nbl):
        w = want[b]
        core = torch.randperm(n, generator=g)[:int(round(w * overlap))].tolist()
        for i in range(R):
            sel = list(core)
            for x in torch.randperm(n, generator=g).tolist():
                if len(sel) >= w:
                    break
                if x not in sel:
                    sel.append(x)
            sel = sorted(sel)
            blocks[b, i, :len(sel)] = torch.tensor(sel, dtype=torch.int32) if sel else blocks[b, i, :0]
            counts[b, i] = len(sel)
    return blocks, counts
