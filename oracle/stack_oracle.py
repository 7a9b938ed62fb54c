"""Float64 CPU oracle of the multi-layer self-speculative decode loop.

TEST INFRASTRUCTURE ONLY.  Only the test-suite may import it.  It shares no
code with the library or its Python package: the seeded inputs (weights,
initial context, first input vector, acceptance draws) are passed in as
arrays, and every attention step calls the float64 functions of vg_oracle.

Sources: [Vegas] "Vegas: Self-Speculative Decoding with Verification-Guided
Sparse Attention" -- "The pith", "Core claim" and Figure 1 (drafting with the
model's own sparse attention over positions chosen by the last verification,
verifying the k + 1 block with full attention, Collect-2-Query capture, the
next selection made from that capture).

The model around the attention path (readings, the pages leave it open):
  layer input   h = bf16(x / sqrt(mean(x^2) + 1e-6))
  projections   q, k, v = bf16(h W_q), bf16(h W_k), bf16(h W_v)   (float64 sum)
  output        o = bf16(attention)   -- the attention path's output type
  residual      x <- x + o
  next token    input of the token after position p = RMS-normalised final
                residual of p (in place of LM head, sampling and embedding)
  acceptance    accepted count = leading ones of the iteration's k draws
Positions: with n tokens cached, draft step t processes position n + t - 1,
writes its K/V there and attends the selection plus [tail_start, n + t); the
verify block is positions n .. n + k (rows attend causally, K/V rewritten);
the selection covers [0, n); then n <- n + a + 1, the next input comes from
verify row a and the next tail starts at the old n.  A one-row verify of the
first token seeds the selections.
"""
from __future__ import annotations

import numpy as np
import torch

from . import vg_oracle as O

RMS_EPS = 1e-6


def bf16(x) -> np.ndarray:
    """Round float64 values to bfloat16 (through float32, round to nearest
    even at each step, as PyTorch's conversion does) and return float64."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64))
    return t.to(torch.bfloat16).to(torch.float64).numpy()


def bf16_stochastic(seed: int):
    """A rounding function to bfloat16 (through float32) that rounds up or
    down at random with probability proportional to the distance from the
    other neighbour: unbiased, every value moves by less than one bf16 ulp.
    Used to measure how far output rounding alone carries the decode loop."""
    rng = np.random.default_rng(seed)

    def rnd(x):
        f = np.ascontiguousarray(x, dtype=np.float64).astype(np.float32)
        bits = f.view(np.uint32)
        low = bits & np.uint32(0xFFFF)
        up = rng.integers(0, 0x10000, size=bits.shape, dtype=np.uint32) < low
        out = (bits & np.uint32(0xFFFF0000)) + (up.astype(np.uint32) << np.uint32(16))
        return out.view(np.float32).astype(np.float64)
    return rnd


def rms_normalise(x):
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + RMS_EPS)


def project(weights_l, x, num_q_heads, num_kv_heads, head_dim):
    """q, k, v of input vectors x [..][H] for one layer: bf16(bf16(rms(x)) W)
    reshaped to [..][heads][d]."""
    h = bf16(rms_normalise(x))
    wq, wk, wv = weights_l
    shp = x.shape[:-1]
    return (bf16(h @ wq).reshape(*shp, num_q_heads, head_dim),
            bf16(h @ wk).reshape(*shp, num_kv_heads, head_dim),
            bf16(h @ wv).reshape(*shp, num_kv_heads, head_dim))


def leading_ones(draws) -> np.ndarray:
    """Accepted draft count per sequence: the length of the leading run of
    True in each row of a [B][k] bool array."""
    d = np.asarray(draws, dtype=bool)
    out = np.zeros(d.shape[0], dtype=np.int64)
    for b in range(d.shape[0]):
        n = 0
        while n < d.shape[1] and d[b, n]:
            n += 1
        out[b] = n
    return out


def decode_stack(weights, contexts, e0, draws, *, num_q_heads, num_kv_heads, head_dim,
                 prefix_lens, n_drafts, top_k, n_sink, n_recent, per_head, iterations, room,
                 record=None, round_out=bf16, force_sets=None):
    """Run the seed verify and `iterations` draft/verify iterations.

    weights  list over layers of (W_q [H][Hq*d], W_k [H][Hkv*d], W_v), float64
    contexts list over layers of (ks, vs), per sequence [Hkv][L_b][d] float64
    e0       [B][H] float64 input vector of the first token
    draws    [iterations][B][k] bool
    record(kind, layer, dict) is called after each attention step with kind
    "seed", "draft" (t = step) or "verify"; verify records carry `out`, the
    captured `rows`, the selection `scores` and `sets`.
    round_out: rounding of attention outputs to bf16 before the residual add
    (round to nearest even; bf16_stochastic gives a perturbed chain).
    force_sets(kind, layer), if given, is called once after each selection
    (after `record` saw it); a non-None result replaces that selection -- to
    run two chains on one sequence of selections.
    Returns the final cache lengths [B]."""
    layers = len(weights)
    B, H = e0.shape
    Hq, Hkv, d = num_q_heads, num_kv_heads, head_dim
    assert Hq * d == H, "the residual adds the attention output: Hq * d must equal H"
    k_ = n_drafts
    scale = 1.0 / np.sqrt(d)
    L0 = [int(L) for L in prefix_lens]
    # dense logical cache per layer and sequence: [Hkv][L_b + room][d]
    K = [[np.zeros((Hkv, L0[b] + room, d)) for b in range(B)] for _ in range(layers)]
    V = [[np.zeros((Hkv, L0[b] + room, d)) for b in range(B)] for _ in range(layers)]
    for l in range(layers):
        for b in range(B):
            K[l][b][:, :L0[b]] = contexts[l][0][b]
            V[l][b][:, :L0[b]] = contexts[l][1][b]

    def qkv(l, x):
        return project(weights[l], x, Hq, Hkv, d)

    def verify_select(l, q, n):
        out, rows = O.verify_attention(q, K[l], V[l], n, scale)
        scores = O.selection_scores(rows, O.CAPTURE_ROWS, Hq, Hkv, per_head)
        sets = O.select_kv(rows, O.CAPTURE_ROWS, n, Hq, Hkv, top_k, n_sink, n_recent, per_head)
        return out, rows, scores, sets

    n = list(L0)
    sets = [None] * layers
    # seed: one-row verify of the first token
    x = e0[:, None, :].copy()
    for l in range(layers):
        q, kk, vv = qkv(l, x)
        for b in range(B):
            K[l][b][:, n[b]] = kk[b, 0]
            V[l][b][:, n[b]] = vv[b, 0]
        out, rows, scores, sets[l] = verify_select(l, q, n)
        if record:
            record("seed", l, dict(out=out, rows=rows, scores=scores, sets=sets[l]))
        forced = force_sets("seed", l) if force_sets is not None else None
        if forced is not None:
            sets[l] = forced
        x = x + round_out(out).reshape(B, 1, H)
    tail_start = list(n)
    n = [m + 1 for m in n]
    e = rms_normalise(x[:, 0])

    for it in range(iterations):
        block = [e]
        for t in range(1, k_ + 1):
            pos = [m + t - 1 for m in n]
            x = block[-1]
            for l in range(layers):
                q, kk, vv = qkv(l, x)
                for b in range(B):
                    K[l][b][:, pos[b]] = kk[b]
                    V[l][b][:, pos[b]] = vv[b]
                out = O.sparse_draft_attention(q, K[l], V[l], sets[l], per_head, tail_start,
                                               [p + 1 for p in pos], scale)
                if record:
                    record("draft", l, dict(out=out, t=t))
                x = x + round_out(out).reshape(B, H)
            block.append(rms_normalise(x))
        X = np.stack(block, axis=1)                       # [B][k+1][H]
        for l in range(layers):
            q, kk, vv = qkv(l, X)
            for b in range(B):
                K[l][b][:, n[b]:n[b] + k_ + 1] = kk[b].transpose(1, 0, 2)
                V[l][b][:, n[b]:n[b] + k_ + 1] = vv[b].transpose(1, 0, 2)
            out, rows, scores, sets[l] = verify_select(l, q, n)
            if record:
                record("verify", l, dict(out=out, rows=rows, scores=scores, sets=sets[l]))
            forced = force_sets("verify", l) if force_sets is not None else None
            if forced is not None:
                sets[l] = forced
            X = X + round_out(out).reshape(B, k_ + 1, H)
        a = leading_ones(draws[it])
        tail_start = list(n)
        e = rms_normalise(X[np.arange(B), a])
        n = [n[b] + int(a[b]) + 1 for b in range(B)]
    return n
