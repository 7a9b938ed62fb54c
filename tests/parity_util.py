"""Helpers for GPU-vs-oracle parity checks.

Tolerances (bf16 inputs/outputs, fp32 accumulation on the GPU, float64 oracle):
  attention outputs   max |gpu - oracle| <= 2e-2 and mean |gpu - oracle| <= 2e-3
  captured logits     |gpu - oracle| <= 1e-3 * max(1, |oracle|)
  index sets          bit-exact against the oracle's fp32 mirror fed the same
                      captured tensor; against the float64 oracle end to end, a
                      position may differ only if its oracle score lies within
                      1e-4 (absolute, on the summed score) of the oracle's
                      top_k-th candidate score.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import vg_oracle as O

OUT_MAX, OUT_MEAN = 2e-2, 2e-3
CAP_REL = 1e-3
GAP = 1e-4


def dense64(inp):
    q = inp.q_verify.double().numpy()
    k = [x.double().numpy() for x in inp.k_dense]
    v = [x.double().numpy() for x in inp.v_dense]
    return q, k, v


def assert_close_out(got, ref, what=""):
    err = np.abs(np.asarray(got, np.float64) - ref)
    assert err.max() <= OUT_MAX, f"{what}: max abs err {err.max():.3e}"
    assert err.mean() <= OUT_MEAN, f"{what}: mean abs err {err.mean():.3e}"
    return float(err.max()), float(err.mean())


def assert_close_capture(got, ref, what=""):
    got = np.asarray(got, np.float64)
    bad = np.abs(got - ref) > CAP_REL * np.maximum(1.0, np.abs(ref))
    assert not bad.any(), f"{what}: {bad.sum()} captured logits out of tolerance, e.g. " \
                          f"{got[bad][:3]} vs {ref[bad][:3]}"


def sub_problem(q, k, v, b, h, g):
    """The verify inputs of one (sequence, KV head): Hq = g, Hkv = 1."""
    return q[b:b + 1, :, h * g:(h + 1) * g], [k[b][h:h + 1]], [v[b][h:h + 1]]


def check_verify(st, inp, pairs=None):
    """Outputs of verify for the (b, kv head) pairs (all if None)."""
    s = inp.spec
    q, k, v = dense64(inp)
    g = s.group
    got = st.out_verify.float().cpu().numpy()
    pairs = pairs or [(b, h) for b in range(s.batch) for h in range(s.num_kv_heads)]
    for b, h in pairs:
        qs, ks, vs = sub_problem(q, k, v, b, h, g)
        out, rows = O.verify_attention(qs, ks, vs, [s.prefix_lens[b]], s.softmax_scale)
        assert_close_out(got[b, :, h * g:(h + 1) * g], out[0], f"verify b={b} h={h}")


def oracle_rows(inp):
    q, k, _ = dense64(inp)
    return O.capture_rows(q, k, inp.spec.prefix_lens, inp.spec.softmax_scale)


def oracle_all(inp):
    """Collect-All capture of the oracle, [B][Hkv][Lmax] float64."""
    q, k, _ = dense64(inp)
    s = inp.spec
    return O.collect_all_sum(q, k, s.prefix_lens, s.softmax_scale, s.num_kv_heads)


GAP_W_REL = 1e-3  # weight scores: near-tie allowance relative to the k-th score


def oracle_weights(inp):
    """VG_CAPTURE_ALL_ROWS of the oracle: (logits [B][Hq][R][Lmax], lse [B][Hq][R])."""
    q, k, _ = dense64(inp)
    return O.capture_all_rows(q, k, inp.spec.prefix_lens, inp.spec.softmax_scale)


def split_all_rows(flat, spec):
    B, Hq, R, Lmax = spec.batch, spec.num_q_heads, spec.n_rows, spec.max_prefix
    a = np.asarray(flat)
    return a[:B * Hq * R * Lmax].reshape(B, Hq, R, Lmax), a[B * Hq * R * Lmax:].reshape(B, Hq, R)


def check_capture(st, inp, rows64):
    s = inp.spec
    cap = st.capture.cpu().numpy()
    if st.capture_mode == O.CAPTURE_ALL_ROWS:
        lg, ls = split_all_rows(cap, s)
        olg, ols = oracle_weights(inp)
        for b, L in enumerate(s.prefix_lens):
            assert_close_capture(lg[b, :, :, :L], olg[b, :, :, :L], f"all-rows logits b={b}")
            assert_close_capture(ls[b], ols[b], f"row lse b={b}")
        return
    if st.capture_mode == O.CAPTURE_ALL_SUM:
        A = oracle_all(inp)
        for b, L in enumerate(s.prefix_lens):
            assert_close_capture(cap[b, :, :L], A[b, :, :L], f"collect-all b={b}")
    elif st.capture_mode == O.CAPTURE_ROWS:
        for b, L in enumerate(s.prefix_lens):
            assert_close_capture(cap[b, :, :, :L], rows64[b, :, :, :L], f"rows b={b}")
    else:
        G = O.group_sum(rows64, s.num_kv_heads)
        for b, L in enumerate(s.prefix_lens):
            assert_close_capture(cap[b, :, :L], G[b, :, :L], f"group sum b={b}")


def gpu_sets(st):
    idx, cnt = st.indices.cpu().numpy(), st.counts.cpu().numpy()
    B, rows, cap = idx.shape
    sets = []
    for b in range(B):
        sets.append([idx[b, r, :cnt[b, r]] for r in range(rows)])
        for r in range(rows):
            assert (idx[b, r, cnt[b, r]:] == -1).all(), "padding must be -1"
    return sets


def check_select_synthetic(spec, capture_mode, per_head, seed=5, device="cuda"):
    """GPU selector vs the oracle's fp32 mirror, both fed the same
    generator-made capture (with many exact ties): bit-exact index sets."""
    from self_speculative_sparse_vg_gb300 import vg
    from self_speculative_sparse_vg_gb300.workloads import make_capture
    cap_cpu = make_capture(spec, capture_mode, seed)
    rows = spec.num_kv_heads if per_head else 1
    capn = min(spec.max_prefix, spec.n_sel_max)
    idx = torch.full((spec.batch, rows, capn), -7, dtype=torch.int32, device=device)
    cnt = torch.zeros(spec.batch, rows, dtype=torch.int32, device=device)
    lens = torch.tensor(spec.prefix_lens, dtype=torch.int32, device=device)
    flag = torch.zeros(1, dtype=torch.int32, device=device)
    vg.select_kv(cap_cpu.to(device), capture_mode, lens, spec.num_q_heads, spec.num_kv_heads,
                 spec.max_prefix, spec.top_k, spec.n_sink, spec.n_recent, per_head, idx, cnt, flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    ref = O.select_kv(cap_cpu.numpy(), capture_mode, spec.prefix_lens, spec.num_q_heads,
                      spec.num_kv_heads, spec.top_k, spec.n_sink, spec.n_recent, per_head,
                      mirror=True)
    got_i, got_c = idx.cpu().numpy(), cnt.cpu().numpy()
    for b in range(spec.batch):
        for r in range(rows):
            n = got_c[b, r]
            assert got_i[b, r, :n].tolist() == ref[b][r].tolist(), f"select b={b} row={r}"
            assert (got_i[b, r, n:] == -1).all(), "padding must be -1"


def _weight_sets_scores(inp, per_head):
    s = inp.spec
    olg, ols = oracle_weights(inp)
    sc = O.weight_scores(olg, ols, s.num_kv_heads, per_head)
    sets = O.select_kv_weights(olg, ols, s.prefix_lens, s.num_kv_heads, s.top_k, s.n_sink,
                               s.n_recent, per_head)
    return sets, sc


def _oracle_capture(inp, rows64, capture_mode):
    """The oracle's capture for a capture mode: Collect-All sums, or the raw
    rows (from which the Collect-2 group sums follow)."""
    if capture_mode == O.CAPTURE_ALL_SUM:
        return oracle_all(inp), O.CAPTURE_ALL_SUM
    return rows64, O.CAPTURE_ROWS


def oracle_sets(inp, rows64, per_head, capture_mode=O.CAPTURE_GROUP_SUM):
    s = inp.spec
    if capture_mode == O.CAPTURE_ALL_ROWS:
        return _weight_sets_scores(inp, per_head)[0]
    cap, mode = _oracle_capture(inp, rows64, capture_mode)
    return O.select_kv(cap, mode, s.prefix_lens, s.num_q_heads, s.num_kv_heads,
                       s.top_k, s.n_sink, s.n_recent, per_head)


def check_select_end_to_end(st, inp, rows64):
    """GPU capture -> GPU select vs float64 oracle capture -> float64 select."""
    s = inp.spec
    gap_rel = False
    if st.capture_mode == O.CAPTURE_ALL_ROWS:
        ref, sc = _weight_sets_scores(inp, st.per_head)
        gap_rel = True
    else:
        cap, mode = _oracle_capture(inp, rows64, st.capture_mode)
        sc = O.selection_scores(cap, mode, s.num_q_heads, s.num_kv_heads, st.per_head)
        ref = O.select_kv(cap, mode, s.prefix_lens, s.num_q_heads, s.num_kv_heads,
                          s.top_k, s.n_sink, s.n_recent, st.per_head)
    got = gpu_sets(st)
    worst = 0.0
    for b, L in enumerate(s.prefix_lens):
        for r in range(len(ref[b])):
            a, o = set(got[b][r].tolist()), set(ref[b][r].tolist())
            if a == o:
                continue
            cand = np.arange(s.n_sink, L - s.n_recent)
            order = np.lexsort((cand, -sc[b, r, cand]))
            kth = sc[b, r, cand[order[s.top_k - 1]]]
            for pos in a ^ o:
                gap = abs(sc[b, r, pos] - kth)
                worst = max(worst, gap)
                lim = GAP_W_REL * abs(kth) if gap_rel else GAP
                assert gap < lim, f"b={b} row={r} pos={pos}: score gap {gap:.3e} to the k-th"
    return worst


def check_drafts(st, inp, oracle_sel, pairs=None, steps=None, min_pairs=1):
    """GPU drafts (run on the GPU's own selection) vs the oracle's drafts on
    the oracle's selection, for the (sequence, KV head) pairs whose two
    selections are identical; at least `min_pairs` pairs must be compared.
    Returns the number of pairs compared."""
    s = inp.spec
    _, k, v = dense64(inp)
    g = s.group
    steps = steps or list(range(1, s.n_drafts + 1))
    pairs = pairs or [(b, h) for b in range(s.batch) for h in range(s.num_kv_heads)]
    mine = gpu_sets(st)
    same = [(b, h) for b, h in pairs
            if mine[b][h if st.per_head else 0].tolist() == oracle_sel[b][h if st.per_head else 0].tolist()]
    for t in steps:
        dq = inp.draft_q[t - 1].double().numpy()
        got = st.out_draft[t - 1].float().cpu().numpy()
        for b, h in same:
            sel = [[oracle_sel[b][h if st.per_head else 0]]]
            ref = O.sparse_draft_attention(dq[b:b + 1, h * g:(h + 1) * g], [k[b][h:h + 1]],
                                           [v[b][h:h + 1]], sel, False, [s.prefix_lens[b]],
                                           [s.prefix_lens[b] + t], s.softmax_scale)
            assert_close_out(got[b, h * g:(h + 1) * g], ref[0], f"draft t={t} b={b} h={h}")
    assert len(same) >= min_pairs, f"only {len(same)} of {len(pairs)} pairs had the oracle's selection"
    return len(same)


def check_drafts_synthetic(st, inp, per_head, seed=9, pairs=None, steps=None):
    """GPU sparse draft vs the oracle, both fed the same generator-made index
    lists (the GPU selection in `st` is overwritten)."""
    from self_speculative_sparse_vg_gb300.workloads import make_selection
    s = inp.spec
    idx, cnt = make_selection(s, per_head, seed)
    st.indices.copy_(idx.to(st.indices.device))
    st.counts.copy_(cnt.to(st.counts.device))
    if st.slots is not None:
        st.slots.copy_(cache_slots(idx, cnt, inp.page_table).to(st.slots.device))
    steps = steps or list(range(1, s.n_drafts + 1))
    for t in steps:
        st.draft(t)
    torch.cuda.synchronize()
    assert int(st.error_flag.item()) == 0
    _, k, v = dense64(inp)
    g = s.group
    pairs = pairs or [(b, h) for b in range(s.batch) for h in range(s.num_kv_heads)]
    sel = [[idx[b, r, :cnt[b, r]].numpy() for r in range(idx.shape[1])] for b in range(s.batch)]
    for t in steps:
        dq = inp.draft_q[t - 1].double().numpy()
        got = st.out_draft[t - 1].float().cpu().numpy()
        for b, h in pairs:
            ref = O.sparse_draft_attention(dq[b:b + 1, h * g:(h + 1) * g], [k[b][h:h + 1]],
                                           [v[b][h:h + 1]], [[sel[b][h if per_head else 0]]], False,
                                           [s.prefix_lens[b]], [s.prefix_lens[b] + t],
                                           s.softmax_scale)
            assert_close_out(got[b, h * g:(h + 1) * g], ref[0], f"draft t={t} b={b} h={h}")


def cache_slots(idx, cnt, page_table):
    """Cache slots of index lists (page-table layout, not method arithmetic):
    page_table[b][p // 16] * 16 + p % 16 for every listed position p, -1
    past the count."""
    idx = idx.long()
    B, rows, cap = idx.shape
    pos = idx.clamp(min=0)
    phys = torch.gather(page_table.long()[:, None, :].expand(B, rows, -1), 2, pos // 16)
    out = phys * 16 + pos % 16
    live = torch.arange(cap)[None, None, :] < cnt.long()[:, :, None]
    return torch.where(live, out, torch.full_like(out, -1)).to(torch.int32)


def check_slots(st, inp):
    """The cache slots the selector wrote beside its positions equal the page
    table's translation of those positions, bit for bit (-1 past the count)."""
    if st.slots is None:
        return
    want = cache_slots(st.indices.cpu(), st.counts.cpu(), inp.page_table)
    got = st.slots.cpu()
    assert torch.equal(got, want), f"{(got != want).sum().item()} cache slots differ"


def poison_draft_workspace(st):
    """NaN bit patterns over the draft workspace (the draft needs none: its
    segments merge inside their cluster, so this must change nothing)."""
    st.ws_draft.fill_(0xFF)


def flag(st):
    torch.cuda.synchronize()
    return int(st.error_flag.item())
