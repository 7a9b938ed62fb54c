"""Pins of the float64 oracle against things other than itself: textbook
causal attention built a different way (full masked score matrix + library
softmax + repeat-KV), closed forms, hand-derived fixtures, brute-force
subset enumeration, and invariants.  CPU only."""
import itertools
import json
import math
import os

import numpy as np
import pytest
from scipy.special import softmax as sp_softmax

from oracle import vg_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_case(rng, B, R, Hq, Hkv, d, Ls):
    q = rng.standard_normal((B, R, Hq, d))
    k = [rng.standard_normal((Hkv, L + R, d)) for L in Ls]
    v = [rng.standard_normal((Hkv, L + R, d)) for L in Ls]
    return q, k, v


def _causal_lm_block(q, kb, vb, L, scale):
    """Textbook causal self-attention of a sequence of length n = L + R, read
    off at the last R query positions.  GQA is expanded by repeating each KV
    head g times (the usual repeat-KV); the mask is the lower triangle."""
    R, Hq, d = q.shape
    Hkv, n, _ = kb.shape
    g = Hq // Hkv
    K = np.repeat(kb, g, axis=0)            # [Hq][n][d]
    V = np.repeat(vb, g, axis=0)
    out = np.empty((R, Hq, d))
    mask = np.tril(np.ones((n, n), dtype=bool))[L:L + R]   # query positions L..L+R-1
    for h in range(Hq):
        S = scale * q[:, h, :] @ K[h].T                    # [R][n]
        S = np.where(mask, S, -np.inf)
        out[:, h, :] = sp_softmax(S, axis=1) @ V[h]
    return out


@pytest.mark.parametrize("R,Hq,Hkv,d,Ls", [
    (1, 4, 4, 4, [1, 9]),        # k = 0: plain decode, MHA
    (3, 4, 1, 8, [5]),           # MQA
    (5, 8, 2, 16, [33, 2]),      # GQA g=4, ragged batch
    (4, 6, 3, 4, [17]),          # g=2
])
def test_verify_equals_causal_lm_attention(R, Hq, Hkv, d, Ls):
    rng = np.random.default_rng(7)
    q, k, v = _rand_case(rng, len(Ls), R, Hq, Hkv, d, Ls)
    scale = 0.37
    out, rows = O.verify_attention(q, k, v, Ls, scale)
    for b, L in enumerate(Ls):
        ref = _causal_lm_block(q[b], k[b], v[b], L, scale)
        np.testing.assert_allclose(out[b], ref, rtol=0, atol=1e-12)
        # captured rows are entries of the same full score matrix
        K = np.repeat(k[b], Hq // Hkv, axis=0)
        for h in range(Hq):
            full0 = scale * K[h] @ q[b, 0, h]
            fullk = scale * K[h] @ q[b, R - 1, h]
            np.testing.assert_allclose(rows[b, h, 0, :L], full0[:L], atol=1e-12)
            np.testing.assert_allclose(rows[b, h, 1, :L], fullk[:L], atol=1e-12)
            assert np.isnan(rows[b, h, :, L:]).all()


def test_verify_capture_golden():
    with open(os.path.join(GOLDEN, "verify_capture_small.json")) as f:
        gd = json.load(f)
    k = np.array(gd["k"], float)[None]          # Hkv = 1
    v = np.array(gd["v"], float)[None]
    q = np.array(gd["q"], float)[None]          # [1][R][Hq][d]
    out, rows = O.verify_attention(q, [k], [v], [gd["prefix_len"]], gd["scale"])
    np.testing.assert_array_equal(rows[0], np.array(gd["rows"]))
    np.testing.assert_array_equal(O.group_sum(rows, 1)[0, 0], np.array(gd["group_sum"]))
    # closed-form outputs: head0 row0 sees positions 0..2 with logits 1,0,1
    e = math.e
    np.testing.assert_allclose(out[0, 0, 0], [e / (2 * e + 1), 1 / (2 * e + 1)], atol=1e-15)
    # head1 bonus row sees 0..3 with logits -1, 1, 0, -2  (0.5*q.k, q=(-2,2))
    w = np.exp([-1.0, 1.0, 0.0, -2.0])
    w /= w.sum()
    np.testing.assert_allclose(out[0, 1, 1], w[0] * np.array([1, 0]) + w[1] * np.array([0, 1])
                               + w[3] * np.array([3, 3]), atol=1e-15)


def test_verify_two_keys_logistic():
    # L = 1, one row: the row attends positions 0 and 1 only.
    q = np.array([1.0, 0.0]).reshape(1, 1, 1, 2)
    k = np.array([[[3.0, 0.0], [1.0, 5.0], [9.0, 9.0]]])   # position 2 is outside the mask
    v = np.array([[[2.0, -1.0], [0.0, 4.0], [100.0, 100.0]]])
    out, _ = O.verify_attention(q, [k], [v], [1], 1.0)
    w0 = 1.0 / (1.0 + math.exp(-(3.0 - 1.0)))
    np.testing.assert_allclose(out[0, 0, 0], w0 * np.array([2, -1]) + (1 - w0) * np.array([0, 4]),
                               atol=1e-15)


def test_verify_constant_keys_mean_v_and_dominant_key():
    rng = np.random.default_rng(3)
    L, R, d = 20, 3, 8
    k = np.tile(rng.standard_normal(d), (1, L + R, 1))
    v = rng.standard_normal((1, L + R, d))
    q = rng.standard_normal((1, R, 2, d))
    out, _ = O.verify_attention(q, [k], [v], [L], 0.5)
    for i in range(R):
        np.testing.assert_allclose(out[0, i, :], np.tile(v[0, :L + i + 1].mean(0), (2, 1)),
                                   atol=1e-12)
    k2 = rng.standard_normal((1, L + R, d)) * 0.01
    k2[0, 7] = 50.0 * q[0, :, 0].mean(0) / np.linalg.norm(q[0, :, 0].mean(0))
    q2 = np.repeat(q[:, :, :1], 2, axis=2)
    q2[0, :, :, :] = k2[0, 7] / 10.0
    out2, _ = O.verify_attention(q2, [k2], [v], [L], 1.0)
    np.testing.assert_allclose(out2[0, :, 0], np.tile(v[0, 7], (R, 1)), atol=1e-9)


def test_verify_affine_in_v_and_mask_boundary():
    rng = np.random.default_rng(5)
    Ls, R = [13], 4
    q, k, v = _rand_case(rng, 1, R, 4, 2, 8, Ls)
    out, _ = O.verify_attention(q, k, v, Ls, 0.3)
    c = rng.standard_normal(8)
    out_shift, _ = O.verify_attention(q, k, [v[0] * 2.0 + c], Ls, 0.3)
    np.testing.assert_allclose(out_shift, 2.0 * out + c, atol=1e-12)
    L = Ls[0]
    for i in range(R):
        # positions beyond L + i must not matter for row i ...
        k_after = k[0].copy()
        v_after = v[0].copy()
        k_after[:, L + i + 1:] += 5.0
        v_after[:, L + i + 1:] -= 7.0
        o2, _ = O.verify_attention(q, [k_after], [v_after], Ls, 0.3)
        np.testing.assert_array_equal(o2[0, i], out[0, i])
        # ... and position L + i (the row's own token) must.
        v_own = v[0].copy()
        v_own[:, L + i] += 1.0
        o3, _ = O.verify_attention(q, k, [v_own], Ls, 0.3)
        assert np.abs(o3[0, i] - out[0, i]).min() > 1e-6


def test_verify_gqa_head_mapping():
    rng = np.random.default_rng(9)
    Hq, Hkv, d, L, R = 8, 2, 4, 10, 2
    q = rng.standard_normal((1, R, Hq, d))
    k = [rng.standard_normal((Hkv, L + R, d))]
    v = [np.stack([np.full((L + R, d), float(h)) for h in range(Hkv)])]
    out, _ = O.verify_attention(q, k, v, [L], 1.0)
    for h in range(Hq):
        np.testing.assert_allclose(out[0, :, h], h // (Hq // Hkv), atol=1e-12)


def test_group_sum_head_grouping():
    B, Hq, Hkv, L = 1, 8, 2, 3
    rows = np.zeros((B, Hq, 2, L))
    for qh in range(Hq):
        rows[0, qh, 0] = qh + 1
        rows[0, qh, 1] = 100 * (qh + 1)
    G = O.group_sum(rows, Hkv)
    np.testing.assert_array_equal(G[0, 0], 101 * (1 + 2 + 3 + 4))
    np.testing.assert_array_equal(G[0, 1], 101 * (5 + 6 + 7 + 8))
    np.testing.assert_array_equal(O.group_sum_mirror(rows, Hkv), G.astype(np.float32))


def test_mirror_summation_order():
    # fp32: (1e8 + 1) -> 1e8 ; (-1e8 + 1) -> -1e8 ; 1e8 + -1e8 = 0.  float64 gives 2.
    rows = np.array([[[[1e8], [1.0]], [[-1e8], [1.0]]]])       # [1][Hq=2][2][L=1]
    assert O.group_sum_mirror(rows, 1)[0, 0, 0] == np.float32(0.0)
    assert O.group_sum(rows, 1)[0, 0, 0] == 2.0
    # head order for the head-averaged score: (1e8 + 1) + -1e8 = 0 in fp32
    G = np.array([[[1e8], [1.0], [-1e8]]], dtype=np.float32)
    s = O.selection_scores(G, O.CAPTURE_GROUP_SUM, 3, 3, per_head=False, mirror=True)
    assert s[0, 0, 0] == np.float32(0.0)
    s64 = O.selection_scores(G, O.CAPTURE_GROUP_SUM, 3, 3, per_head=False, mirror=False)
    assert s64[0, 0, 0] == 1.0


def test_select_golden_ties():
    with open(os.path.join(GOLDEN, "select_ties.json")) as f:
        gd = json.load(f)
    got = O.select_row(np.array(gd["scores"], float), gd["prefix_len"], gd["top_k"],
                       gd["n_sink"], gd["n_recent"])
    assert got.tolist() == gd["expected"]


def _brute_force_select(score, L, top_k, n_sink, n_recent):
    """Max-sum subset of the candidates; among max-sum subsets the
    lexicographically smallest (= ties to lower positions)."""
    cand = list(range(n_sink, L - n_recent))
    best = None
    for sub in itertools.combinations(cand, top_k):
        key = (-sum(score[j] for j in sub), sub)
        if best is None or key < best:
            best = key
    return sorted(list(range(n_sink)) + list(best[1]) + list(range(L - n_recent, L)))


def test_select_matches_subset_enumeration():
    rng = np.random.default_rng(11)
    for trial in range(60):
        L = int(rng.integers(6, 15))
        n_sink = int(rng.integers(0, 3))
        n_recent = int(rng.integers(0, 3))
        top_k = int(rng.integers(1, max(2, L - n_sink - n_recent)))
        score = rng.integers(-3, 4, L).astype(float)        # many ties
        got = O.select_row(score, L, top_k, n_sink, n_recent)
        if L <= n_sink + n_recent + top_k:
            assert got.tolist() == list(range(L))
        else:
            assert got.tolist() == _brute_force_select(score, L, top_k, n_sink, n_recent)


def test_select_structure_and_small_prefix():
    rng = np.random.default_rng(2)
    L, top_k, ns, nr = 500, 40, 4, 16
    s = rng.standard_normal(L)
    got = O.select_row(s, L, top_k, ns, nr)
    assert len(got) == ns + nr + top_k and (np.diff(got) > 0).all()
    assert set(range(ns)) <= set(got.tolist()) and set(range(L - nr, L)) <= set(got.tolist())
    # every kept candidate scores >= every dropped candidate
    kept = [j for j in got if ns <= j < L - nr]
    dropped = [j for j in range(ns, L - nr) if j not in set(kept)]
    assert s[kept].min() >= s[dropped].max()
    assert O.select_row(s, 60, 40, 4, 16).tolist() == list(range(60))
    assert O.select_row(s, 3, 40, 4, 16).tolist() == [0, 1, 2]


def test_select_mirror_equals_float64_on_exact_inputs():
    rng = np.random.default_rng(4)
    B, Hq, Hkv, L = 2, 8, 2, 300
    rows = rng.integers(-50, 50, (B, Hq, 2, L)).astype(np.float64)
    for per_head in (False, True):
        a = O.select_kv(rows, O.CAPTURE_ROWS, [L, L - 37], Hq, Hkv, 20, 4, 8, per_head, mirror=False)
        m = O.select_kv(rows, O.CAPTURE_ROWS, [L, L - 37], Hq, Hkv, 20, 4, 8, per_head, mirror=True)
        for b in range(B):
            for r in range(len(a[b])):
                assert a[b][r].tolist() == m[b][r].tolist()
    # head order does not change the head-averaged set on exact inputs
    G = O.group_sum(rows, Hkv)
    s1 = O.select_kv(G, O.CAPTURE_GROUP_SUM, [L, L], Hq, Hkv, 20, 4, 8, False)
    s2 = O.select_kv(G[:, ::-1].copy(), O.CAPTURE_GROUP_SUM, [L, L], Hq, Hkv, 20, 4, 8, False)
    assert all(x[0].tolist() == y[0].tolist() for x, y in zip(s1, s2))


def test_planted_heavy_hitters_recovered():
    """Seeded 2K-context workload with 16 keys planted along the group's query
    direction: verify capture + head-averaged selection must keep all 16."""
    from self_speculative_sparse_vg_gb300.workloads import WORKLOADS, make_inputs
    spec = WORKLOADS["tiny_d64_2k"]
    inp = make_inputs(spec)
    q = inp.q_verify.double().numpy()
    k = [x.double().numpy() for x in inp.k_dense]
    v = [x.double().numpy() for x in inp.v_dense]
    out, rows = O.verify_attention(q, k, v, spec.prefix_lens, spec.softmax_scale)
    sel = O.select_kv(O.group_sum(rows, spec.num_kv_heads), O.CAPTURE_GROUP_SUM, spec.prefix_lens,
                      spec.num_q_heads, spec.num_kv_heads, spec.top_k, spec.n_sink, spec.n_recent,
                      per_head=False)
    assert set(inp.planted[0].tolist()) <= set(sel[0][0].tolist())
    assert len(sel[0][0]) == spec.n_sel_max
    for per_head in (True,):
        selh = O.select_kv(rows, O.CAPTURE_ROWS, spec.prefix_lens, spec.num_q_heads,
                           spec.num_kv_heads, spec.top_k, spec.n_sink, spec.n_recent, per_head)
        for r in selh[0]:
            assert set(inp.planted[0].tolist()) <= set(r.tolist())


def test_sparse_draft_full_selection_equals_dense():
    rng = np.random.default_rng(21)
    Hq, Hkv, d, L, t = 8, 2, 16, 40, 3
    q = rng.standard_normal((1, Hq, d))
    k = [rng.standard_normal((Hkv, L + t, d))]
    v = [rng.standard_normal((Hkv, L + t, d))]
    cur = L + t
    sel = [[np.arange(L)]]
    out = O.sparse_draft_attention(q, k, v, sel, False, [L], [cur], 0.25)
    # dense decode attention at query position cur-1 (textbook, repeat-KV)
    ref = _causal_lm_block(q[0][None], k[0][:, :cur], v[0][:, :cur], cur - 1, 0.25)[0]
    np.testing.assert_allclose(out[0], ref, atol=1e-12)


def test_sparse_draft_ignores_unselected_and_order():
    rng = np.random.default_rng(22)
    Hq, Hkv, d, L = 4, 2, 8, 50
    q = rng.standard_normal((1, Hq, d))
    k = [rng.standard_normal((Hkv, L + 2, d))]
    v = [rng.standard_normal((Hkv, L + 2, d))]
    sel0 = np.sort(rng.choice(L, 12, replace=False))
    sel1 = np.sort(rng.choice(L, 9, replace=False))
    idx = [[sel0, sel1]]
    out = O.sparse_draft_attention(q, k, v, idx, True, [L], [L + 2], 0.4)
    k2, v2 = k[0].copy(), v[0].copy()
    for h, s in enumerate((sel0, sel1)):
        mask = np.ones(L + 2, bool)
        mask[s] = False
        mask[L:] = False
        k2[h, mask] = 1e3
        v2[h, mask] = -1e3
    out2 = O.sparse_draft_attention(q, [k2], [v2], idx, True, [L], [L + 2], 0.4)
    np.testing.assert_array_equal(out, out2)
    out3 = O.sparse_draft_attention(q, k, v, [[sel0[::-1], sel1[::-1]]], True, [L], [L + 2], 0.4)
    np.testing.assert_allclose(out3, out, atol=1e-13)
    # empty selection: one tail token -> its V row
    out4 = O.sparse_draft_attention(q, k, v, [[np.array([], int), np.array([], int)]], True,
                                    [L], [L + 1], 0.4)
    for h in range(Hq):
        np.testing.assert_allclose(out4[0, h], v[0][h // 2, L], atol=1e-15)


def test_paging_round_trip():
    from self_speculative_sparse_vg_gb300.workloads import small_spec, make_inputs
    inp = make_inputs(small_spec(shuffle_pages=True, extra_pages=3))
    for b, kd in enumerate(inp.k_dense):
        n = kd.shape[1]
        npg = (n + 15) // 16
        ids = inp.page_table[b, :npg].long()
        rec = inp.k_pages[ids].permute(1, 0, 2, 3).reshape(kd.shape[0], npg * 16, -1)[:, :n]
        assert (rec == kd).all()
        recv = inp.v_pages[ids].permute(1, 0, 2, 3).reshape(kd.shape[0], npg * 16, -1)[:, :n]
        assert (recv == inp.v_dense[b]).all()
        assert (inp.page_table[b, npg:] == -1).all()


def test_capture_rows_equals_verify_capture():
    rng = np.random.default_rng(31)
    q, k, v = _rand_case(rng, 2, 4, 8, 2, 16, [19, 6])
    _, rows = O.verify_attention(q, k, v, [19, 6], 0.2)
    np.testing.assert_allclose(O.capture_rows(q, k, [19, 6], 0.2), rows, rtol=0, atol=1e-12)


def test_collect_all_with_two_rows_equals_collect_two():
    """With k = 1 the block has only rows 0 and k, so Collect-All and the
    Collect-2 group sum are the same quantity."""
    rng = np.random.default_rng(41)
    q, k, _ = _rand_case(rng, 2, 2, 8, 2, 16, [23, 7])
    A = O.collect_all_sum(q, k, [23, 7], 0.3, 2)
    G = O.group_sum(O.capture_rows(q, k, [23, 7], 0.3), 2)
    np.testing.assert_allclose(A, G, rtol=0, atol=1e-12)


def test_collect_all_is_linear_in_the_rows():
    """Summing logits over rows equals the logit of the summed query: a
    one-row capture of sum_i q_i gives both Collect-2 slots equal to that
    row, so Collect-All = half of its group sum."""
    rng = np.random.default_rng(42)
    q, k, _ = _rand_case(rng, 1, 6, 8, 2, 8, [40])
    A = O.collect_all_sum(q, k, [40], 0.5, 2)
    qs = q.sum(axis=1, keepdims=True)
    G1 = O.group_sum(O.capture_rows(qs, k, [40], 0.5), 2)
    np.testing.assert_allclose(A, G1 / 2, rtol=0, atol=1e-10)
    # it differs from Collect-2 once the block has middle rows
    G2 = O.group_sum(O.capture_rows(q, k, [40], 0.5), 2)
    assert np.abs(A - G2).max() > 1e-3


def test_collect_all_hand_values():
    """d = 1, one KV head with keys [1, -2, 3], two query heads, three rows:
    A_j = scale * k_j * (sum of all six query values)."""
    q = np.array([[[[1.0], [2.0]], [[0.5], [-1.0]], [[4.0], [0.25]]]])   # [1][3][2][1]
    k = [np.array([[[1.0], [-2.0], [3.0], [9.0], [9.0], [9.0]]])]        # [1][6][1]
    A = O.collect_all_sum(q, k, [3], 2.0, 1)
    total = 1 + 2 + 0.5 - 1 + 4 + 0.25
    np.testing.assert_array_equal(A[0, 0], 2.0 * total * np.array([1.0, -2.0, 3.0]))


def test_all_rows_lse_is_logsumexp_of_the_causal_score_matrix():
    from scipy.special import logsumexp
    rng = np.random.default_rng(51)
    q, k, _ = _rand_case(rng, 2, 4, 6, 3, 8, [21, 9])
    logits, lse = O.capture_all_rows(q, k, [21, 9], 0.35)
    for b, L in enumerate([21, 9]):
        Hkv = k[b].shape[0]
        K = np.repeat(k[b], 6 // Hkv, axis=0)          # repeat-KV GQA expansion
        for h in range(6):
            S = 0.35 * q[b, :, h, :] @ K[h].T           # [R][L + R], textbook full scores
            for i in range(4):
                np.testing.assert_allclose(lse[b, h, i], logsumexp(S[i, :L + i + 1]), rtol=1e-12)
                np.testing.assert_allclose(logits[b, h, i, :L], S[i, :L], rtol=0, atol=1e-12)


def test_weight_scores_are_row_normalised_weights():
    """Each row's weights over everything it attends sum to 1, so the prefix
    part plus the (separately computed) block part of the per-head sums is
    exactly the number of window rows; constant keys give 1 / (L + i + 1)."""
    rng = np.random.default_rng(52)
    q, k, _ = _rand_case(rng, 1, 3, 4, 2, 8, [30])
    logits, lse = O.capture_all_rows(q, k, [30], 0.5)
    sc = O.weight_scores(logits, lse, 2, True)           # [1][2][30]
    for h in range(2):
        block = 0.0
        for qh in (2 * h, 2 * h + 1):
            for i in range(3):
                s_blk = 0.5 * (k[0][h, 30:30 + i + 1] @ q[0, i, qh])
                block += np.exp(s_blk - lse[0, qh, i]).sum()
        np.testing.assert_allclose(sc[0, h].sum() + block, 2 * 3, rtol=1e-12)
    kc = [np.ones((2, 33, 8))]
    logits, lse = O.capture_all_rows(q, kc, [30], 0.5)
    sc = O.weight_scores(logits, lse, 2, False)
    want = 4 * sum(1.0 / (30 + i + 1) for i in range(3))
    np.testing.assert_allclose(sc[0, 0], want, rtol=1e-12)


def test_weight_selection_ranks_like_logits_for_one_row_and_head():
    """With one query head and one row, exp(s - lse) is increasing in s, so
    the weight-ranked selection equals the logit-ranked one."""
    rng = np.random.default_rng(53)
    q, k, _ = _rand_case(rng, 2, 1, 1, 1, 16, [200, 77])
    logits, lse = O.capture_all_rows(q, k, [200, 77], 0.25)
    a = O.select_kv_weights(logits, lse, [200, 77], 1, 20, 2, 5, False)
    rows = O.capture_rows(q, k, [200, 77], 0.25)
    b_ = O.select_kv(rows, O.CAPTURE_ROWS, [200, 77], 1, 1, 20, 2, 5, False)
    for x, y in zip(a, b_):
        assert x[0].tolist() == y[0].tolist()


def test_sparse_verify_with_every_block_is_dense_verify():
    """Selecting every prefix block reproduces full verification; selecting
    none leaves only the causal block."""
    rng = np.random.default_rng(61)
    q, k, v = _rand_case(rng, 2, 3, 4, 2, 8, [37, 16])
    full = [[list(range((L + 15) // 16)) for _ in range(3)] for L in (37, 16)]
    dense, _ = O.verify_attention(q, k, v, [37, 16], 0.4)
    np.testing.assert_allclose(O.sparse_verify_attention(q, k, v, [37, 16], full, 0.4), dense,
                               rtol=0, atol=1e-12)
    none = [[[] for _ in range(3)] for _ in range(2)]
    got = O.sparse_verify_attention(q, k, v, [37, 16], none, 0.4)
    # row 0 with no blocks attends only its own position: its V row
    for b, L in enumerate((37, 16)):
        for h in range(4):
            np.testing.assert_allclose(got[b, 0, h], v[b][h // 2, L], rtol=0, atol=1e-12)


def test_sparse_verify_equals_masked_textbook_attention():
    """A brute-force mask over the full causal score matrix."""
    rng = np.random.default_rng(62)
    q, k, v = _rand_case(rng, 1, 4, 2, 1, 8, [70])
    blocks = [[[0, 3], [1], [4, 0, 2], []]]
    got = O.sparse_verify_attention(q, k, v, [70], blocks, 0.3)
    for i in range(4):
        allowed = [j for j in range(70) if j // 16 in blocks[0][i]] + list(range(70, 70 + i + 1))
        for h in range(2):
            S = 0.3 * (k[0][0] @ q[0, i, h])                 # every position of the sequence
            mask = np.full(S.shape, -np.inf)
            mask[allowed] = 0.0
            w = sp_softmax(S + mask)
            np.testing.assert_allclose(got[0, i, h], w @ v[0][0], rtol=0, atol=1e-12)


def test_select_without_top_k_is_sink_and_recent():
    """top_k = 0 keeps exactly [0, n_sink) and [L - n_recent, L), whatever the
    scores; with n_sink = n_recent = 0 the set is the top_k by a plain stable
    sort (score descending, position ascending)."""
    rng = np.random.default_rng(3)
    L = 300
    score = np.round(rng.standard_normal(L), 1)  # many exact ties
    got = O.select_row(score, L, 0, 5, 7)
    assert got.tolist() == list(range(5)) + list(range(L - 7, L))
    order = sorted(range(L), key=lambda j: (-score[j], j))[:40]
    assert O.select_row(score, L, 40, 0, 0).tolist() == sorted(order)
