"""Float64 CPU oracle for verification-guided self-speculative sparse attention.

TEST INFRASTRUCTURE ONLY.  This module is the plain, slow, obviously correct
statement of what the GPU path computes.  Only the test-suite, the smoke check
and the benchmark's CPU-baseline leg may import it; the library itself never
does, and the library shares no code with it.

Sources (page title, then the section / figure on that page):
  [Vegas]  "Vegas: Self-Speculative Decoding with Verification-Guided Sparse
           Attention" (arXiv 2602.07223) -- "The pith", "Core claim", "What
           carries the argument", Figure 1 and Figure 6 captions, Appendix A
           ("Attention Weights vs. Attention Logits").
  [SSL]    "A Sparse Glimpse of the Whole: Train-Free Self-Speculative
           Decoding" (arXiv 2607.27735) -- "Core claim", "What carries the
           argument" (per-head sink + recent + top-ranked index, dense cache
           kept, i.e. recallable).

Conventions (float64 everywhere unless a function says "mirror"):
  q        [B][R][Hq][d]      R = k + 1 verify rows (k drafts plus the bonus
                              position; the bonus token counts as a row).
  k, v     list over b of [Hkv][n_b][d], n_b >= L_b + R: the dense logical
           cache; positions L_b .. L_b+R-1 hold the verify block itself.
  L_b      committed prefix length of sequence b.
  GQA      query head h reads KV head h // g with g = Hq / Hkv.

Readings where the pages are silent (each is listed in the design notes):
  * causal verify block: row i attends positions [0, L_b + i]          (R2)
  * the captured rows are rows 0 and k (first draft, bonus)            (R1)
  * captured value is softmax_scale * q.k before softmax; scale 1
    gives the raw logit qK^T of Appendix A                              (R4)
  * the two rows are summed, heads are summed (rank-equal to the mean) (R5, R6)
  * selection candidates are prefix positions [n_sink, L_b - n_recent);
    ties go to the lower position; output ascending                    (R3, R10, R11)
  * drafting attends the selection plus every position >= tail_start   (R13)
"""
from __future__ import annotations

import numpy as np

CAPTURE_GROUP_SUM = 1   # per-KV-head sum of the two captured rows
CAPTURE_ROWS = 2        # the two raw rows per query head
CAPTURE_ALL_SUM = 3     # per-KV-head sum of every verify row (Collect-All)
CAPTURE_ALL_ROWS = 4    # every row's logits plus its softmax normaliser (weights)


def _softmax_weights(s: np.ndarray) -> np.ndarray:
    """exp(s - max s) / sum exp(s - max s), float64."""
    e = np.exp(s - s.max())
    return e / e.sum()


def verify_attention(q, k, v, prefix_lens, scale):
    """Full-KV verification attention with Collect-2-Query capture.

    [Vegas] "The pith" / "Core claim": the verify pass is ordinary full
    attention over the cache for the k+1 block rows, and it also writes the
    pre-softmax logits of the first draft token (row 0) and of the bonus
    token (row k) for the prefix positions.

    Returns
      out   [B][R][Hq][d]          softmax(scale * q K^T) V over [0, L_b + i]
      rows  [B][Hq][2][Lmax]       rows[b,h,0,j] = scale*q_{b,0,h}.k_j and
                                   rows[b,h,1,j] = scale*q_{b,k,h}.k_j for
                                   j < L_b, NaN beyond L_b.
    """
    B, R, Hq, d = q.shape
    Hkv = k[0].shape[0]
    g = Hq // Hkv
    Lmax = int(max(prefix_lens))
    out = np.zeros((B, R, Hq, d))
    rows = np.full((B, Hq, 2, Lmax), np.nan)
    for b in range(B):
        L = int(prefix_lens[b])
        for h in range(Hq):
            kvh = h // g
            for i in range(R):
                n = L + i + 1
                s = scale * (k[b][kvh, :n] @ q[b, i, h])
                out[b, i, h] = _softmax_weights(s) @ v[b][kvh, :n]
                if i == 0:
                    rows[b, h, 0, :L] = s[:L]
                if i == R - 1:
                    rows[b, h, 1, :L] = s[:L]
    return out, rows


def sparse_verify_attention(q, k, v, prefix_lens, blocks, scale):
    """Sparse verification: every verify row attends its own selection.

    [SSV] section 4.2 and Figures 2/4/5: each verifier query carries its own
    sparse layout; the exact merged schedule changes only how shared blocks
    are loaded, not what each query attends.  Row i of sequence b attends
    the prefix positions of its 16-position blocks and the verify block
    causally: {j < L_b : j // 16 in blocks[b][i]} u [L_b, L_b + i] (R25).

    blocks: list over b of lists over rows of block numbers (any order).
    Returns out [B][R][Hq][d]."""
    B, R, Hq, d = q.shape
    Hkv = k[0].shape[0]
    g = Hq // Hkv
    out = np.zeros((B, R, Hq, d))
    for b in range(B):
        L = int(prefix_lens[b])
        for i in range(R):
            sel = sorted(set(int(x) for x in blocks[b][i]))
            pos = [j for blk in sel for j in range(16 * blk, min(16 * blk + 16, L))]
            att = np.array(pos + list(range(L, L + i + 1)), dtype=np.int64)
            for h in range(Hq):
                kvh = h // g
                s = scale * (k[b][kvh, att] @ q[b, i, h])
                out[b, i, h] = _softmax_weights(s) @ v[b][kvh, att]
    return out


def capture_rows(q, k, prefix_lens, scale):
    """Only the Collect-2-Query rows of verify_attention, for large inputs:
    rows[b,h,0,j] = scale*q_{b,0,h}.k_j and rows[b,h,1,j] = scale*q_{b,k,h}.k_j
    for prefix positions j < L_b (NaN beyond).  [Vegas] "Core claim"."""
    B, R, Hq, d = q.shape
    Hkv = k[0].shape[0]
    g = Hq // Hkv
    Lmax = int(max(prefix_lens))
    rows = np.full((B, Hq, 2, Lmax), np.nan)
    for b in range(B):
        L = int(prefix_lens[b])
        for h in range(Hq):
            kp = k[b][h // g, :L]
            rows[b, h, 0, :L] = scale * (kp @ q[b, 0, h])
            rows[b, h, 1, :L] = scale * (kp @ q[b, R - 1, h])
    return rows


def collect_all_sum(q, k, prefix_lens, scale, num_kv_heads):
    """Collect-All-Query capture: A[b,h,j] = sum over every verify row i and
    every query head of KV head h of scale*q_{b,i,head}.k_j, for prefix
    positions j < L_b (NaN beyond), float64.  [Vegas] Figure 6 and "Core
    claim": the rule that aggregates all rows of the block, which Collect-2
    replaces by its two boundary rows."""
    B, R, Hq, d = q.shape
    g = Hq // num_kv_heads
    Lmax = int(max(prefix_lens))
    A = np.full((B, num_kv_heads, Lmax), np.nan)
    for b in range(B):
        L = int(prefix_lens[b])
        for h in range(num_kv_heads):
            kp = k[b][h, :L]
            acc = np.zeros(L)
            for qh in range(h * g, (h + 1) * g):
                for i in range(R):
                    acc += scale * (kp @ q[b, i, qh])
            A[b, h, :L] = acc
    return A


def capture_all_rows(q, k, prefix_lens, scale):
    """Every verify row's logits and softmax normaliser, for weight
    statistics.  [SSL] "What carries the argument" (the importance signal is
    the attention weights of a window of verification queries; the window
    here is the k+1 block rows).

    Returns logits [B][Hq][R][Lmax] (scale*q.k at prefix positions j < L_b,
    NaN beyond) and lse [B][Hq][R] = ln sum_{j <= L_b + i} exp(scale*q_i.k_j),
    the normaliser of row i over everything it attends (R2)."""
    B, R, Hq, d = q.shape
    Hkv = k[0].shape[0]
    g = Hq // Hkv
    Lmax = int(max(prefix_lens))
    logits = np.full((B, Hq, R, Lmax), np.nan)
    lse = np.zeros((B, Hq, R))
    for b in range(B):
        L = int(prefix_lens[b])
        for h in range(Hq):
            for i in range(R):
                s = scale * (k[b][h // g, :L + i + 1] @ q[b, i, h])
                logits[b, h, i, :L] = s[:L]
                m = s.max()
                lse[b, h, i] = m + np.log(np.exp(s - m).sum())
    return logits, lse


def weight_scores(logits, lse, num_kv_heads, per_head):
    """Selection score from post-softmax weights: for each prefix position,
    the sum over the selection row's query heads and all window rows of
    exp(logit - lse).  [SSL] "What carries the argument"; a sum ranks like
    the mean.  Returns [B][1 or Hkv][Lmax] float64."""
    B, Hq, R, Lmax = logits.shape
    g = Hq // num_kv_heads
    w = np.exp(logits - lse[..., None])              # [B][Hq][R][Lmax]
    per_q = w.sum(axis=2)                            # [B][Hq][Lmax]
    G = per_q.reshape(B, num_kv_heads, g, Lmax).sum(axis=2)
    return G if per_head else G.sum(axis=1, keepdims=True)


def select_kv_weights(logits, lse, prefix_lens, num_kv_heads, top_k, n_sink, n_recent, per_head):
    """Index sets from weight_scores, by select_row."""
    sc = weight_scores(logits, lse, num_kv_heads, per_head)
    return [[select_row(sc[b, r], L, top_k, n_sink, n_recent) for r in range(sc.shape[1])]
            for b, L in enumerate(prefix_lens)]


def group_sum(rows, num_kv_heads):
    """G[b,h,j] = sum over the query heads q of KV head h of
    (row0[q,j] + rowk[q,j]), float64.  [Vegas] "What carries the argument":
    the two captured rows are aggregated across the heads."""
    B, Hq, _, Lmax = rows.shape
    g = Hq // num_kv_heads
    pair = rows[:, :, 0, :] + rows[:, :, 1, :]
    return pair.reshape(B, num_kv_heads, g, Lmax).sum(axis=2)


def group_sum_mirror(rows, num_kv_heads):
    """Same as group_sum in float32 with one fixed order, the order the GPU
    selector and capture epilogue use: for each KV head h,
    acc = (r0[q0] + rk[q0]); acc = acc + (r0[q1] + rk[q1]); ... ascending q."""
    r = np.asarray(rows, dtype=np.float32)
    B, Hq, _, Lmax = r.shape
    g = Hq // num_kv_heads
    G = np.empty((B, num_kv_heads, Lmax), dtype=np.float32)
    for h in range(num_kv_heads):
        acc = r[:, h * g, 0, :] + r[:, h * g, 1, :]
        for qi in range(1, g):
            qh = h * g + qi
            acc = acc + (r[:, qh, 0, :] + r[:, qh, 1, :])
        G[:, h, :] = acc
    return G


def selection_scores(capture, capture_mode, num_q_heads, num_kv_heads, per_head, mirror=False):
    """Per-position ranking score of the verification-guided selector.

    [Vegas] "Core claim": average the captured logits across the attention
    heads (a sum ranks identically), one score per prefix position.
    [SSL] "What carries the argument": per-head variant, here one score per
    KV head (the unit at which GQA loads KV).

    capture: GROUP_SUM or ALL_SUM -> [B][Hkv][Lmax];  ROWS -> [B][Hq][2][Lmax]
    returns  [B][1 or Hkv][Lmax]  (float64, or float32 when mirror)
    """
    if capture_mode == CAPTURE_ROWS:
        G = group_sum_mirror(capture, num_kv_heads) if mirror else group_sum(capture, num_kv_heads)
    elif capture_mode in (CAPTURE_GROUP_SUM, CAPTURE_ALL_SUM):
        G = np.asarray(capture, dtype=np.float32 if mirror else np.float64)
    else:
        raise ValueError("capture_mode")
    if per_head:
        return G
    if mirror:
        acc = G[:, 0, :].copy()
        for h in range(1, num_kv_heads):
            acc = acc + G[:, h, :]
        return acc[:, None, :]
    return G.sum(axis=1, keepdims=True)


def select_row(score, L, top_k, n_sink, n_recent):
    """Sink + recent + top-k index set for one selection row.

    [SSL] "What carries the argument": sink tokens, recent tokens and the
    top-ranked historical tokens.  [Vegas] "Core claim": the top-k prefix
    positions by combined score.  Candidates are [n_sink, L - n_recent);
    the k best by (score descending, position ascending) are kept.  When the
    prefix is no longer than the budget every position is kept.
    Returns the ascending int64 array of selected positions.
    """
    L = int(L)
    if L <= n_sink + n_recent + top_k:
        return np.arange(L, dtype=np.int64)
    cand = np.arange(n_sink, L - n_recent, dtype=np.int64)
    sc = np.asarray(score[n_sink:L - n_recent], dtype=np.float64)
    order = np.lexsort((cand, -sc))          # primary: -score, secondary: position
    chosen = cand[order[:top_k]]
    return np.sort(np.concatenate([np.arange(n_sink, dtype=np.int64), chosen,
                                   np.arange(L - n_recent, L, dtype=np.int64)]))


def select_kv(capture, capture_mode, prefix_lens, num_q_heads, num_kv_heads,
              top_k, n_sink, n_recent, per_head, mirror=False):
    """Verification-guided KV selection for every (sequence, row).
    Returns a list over b of lists over rows (1 or Hkv) of index arrays."""
    sc = selection_scores(capture, capture_mode, num_q_heads, num_kv_heads, per_head, mirror)
    res = []
    for b, L in enumerate(prefix_lens):
        res.append([select_row(sc[b, r], L, top_k, n_sink, n_recent) for r in range(sc.shape[1])])
    return res


def sparse_draft_attention(q, k, v, indices, per_head, tail_start, cur_len, scale):
    """Sparse decode attention of one draft position per sequence.

    [Vegas] "Core claim" and Figure 1: the draft token attends only the
    selected KV entries; the tokens generated since the selection (the dense
    tail [tail_start, cur_len), including the query's own entry) are
    attended as well.  softmax(scale q K_A^T) V_A over A = Sel u tail.

    q: [B][Hq][d];  indices[b][row] ascending positions < tail_start[b].
    returns out [B][Hq][d]
    """
    B, Hq, d = q.shape
    Hkv = k[0].shape[0]
    g = Hq // Hkv
    out = np.zeros((B, Hq, d))
    for b in range(B):
        tail = np.arange(int(tail_start[b]), int(cur_len[b]), dtype=np.int64)
        for h in range(Hq):
            kvh = h // g
            sel = np.asarray(indices[b][kvh if per_head else 0], dtype=np.int64)
            att = np.concatenate([sel, tail])
            s = scale * (k[b][kvh, att] @ q[b, h])
            out[b, h] = _softmax_weights(s) @ v[b][kvh, att]
    return out
