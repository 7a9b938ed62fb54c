"""Pins of the float64 decode-loop oracle (oracle/stack_oracle.py) to facts
that do not depend on it:

* With a selection budget that covers every cached position, drafting is
  dense attention, so every draft step must reproduce -- at every layer --
  the verify row of the same position (row t-1 for draft step t).  Any slip
  in positions, tail bounds, K/V writes, block assembly or the residual chain
  breaks this equality.
* With a small budget the same comparison must fail (the pin is not vacuous).
* The accepted count is the length of the leading run of accepted drafts;
  entries after the first rejection do not matter, and the cache grows by
  accepted + 1 tokens per iteration.
* The seed row and the first verify are plain causal softmax attention,
  checked by a brute-force loop over positions.
"""
import itertools
import math

import numpy as np
import pytest

from oracle import stack_oracle as SO


def _inputs(layers=2, H=32, Hq=4, Hkv=2, d=8, lens=(5, 9), k=3, iters=3, seed=0):
    rng = np.random.default_rng(seed)
    w = [tuple(SO.bf16(rng.standard_normal((H, n * d)) / math.sqrt(H)) for n in (Hq, Hkv, Hkv))
         for _ in range(layers)]
    ctx = [([SO.bf16(rng.standard_normal((Hkv, L, d))) for L in lens],
            [SO.bf16(rng.standard_normal((Hkv, L, d))) for L in lens]) for _ in range(layers)]
    e0 = rng.standard_normal((len(lens), H))
    draws = rng.random((iters, len(lens), k)) < 0.6
    return w, ctx, e0, draws


def _run(top_k, n_sink=1, n_recent=2, per_head=False, **kw):
    k = kw.get("k", 3)
    iters = kw.get("iters", 3)
    lens = kw.get("lens", (5, 9))
    w, ctx, e0, draws = _inputs(**kw)
    recs = []
    n = SO.decode_stack(w, ctx, e0, draws, num_q_heads=kw.get("Hq", 4),
                        num_kv_heads=kw.get("Hkv", 2), head_dim=kw.get("d", 8), prefix_lens=lens,
                        n_drafts=k, top_k=top_k, n_sink=n_sink, n_recent=n_recent,
                        per_head=per_head, iterations=iters, room=1 + (iters + 1) * (k + 1),
                        record=lambda kind, l, r: recs.append((kind, l, r)))
    return recs, n, draws, (w, ctx, e0)


def _draft_vs_verify(recs, layers, k):
    """Max |draft step t output - verify row t-1 output| over the run."""
    worst = 0.0
    drafts = {}
    it = 0
    for kind, l, r in recs:
        if kind == "draft":
            drafts[(r["t"], l)] = r["out"]
        elif kind == "verify":
            for t in range(1, k + 1):
                worst = max(worst, float(np.abs(drafts[(t, l)] - r["out"][:, t - 1]).max()))
            if l == layers - 1:
                drafts = {}
                it += 1
    return worst, it


@pytest.mark.parametrize("per_head", [False, True])
def test_full_budget_drafts_equal_verify_rows(per_head):
    recs, _, _, _ = _run(top_k=1000, per_head=per_head)
    worst, iters = _draft_vs_verify(recs, layers=2, k=3)
    assert iters == 3
    assert worst < 1e-12, worst


def test_small_budget_drafts_differ_from_verify_rows():
    recs, _, _, _ = _run(top_k=1, n_sink=1, n_recent=1, lens=(40, 57))
    worst, _ = _draft_vs_verify(recs, layers=2, k=3)
    assert worst > 1e-3, worst


def test_leading_ones_and_length_bookkeeping():
    k = 4
    for bits in itertools.product([False, True], repeat=k):
        a = SO.leading_ones(np.array([bits]))[0]
        first_false = bits.index(False) if False in bits else k
        assert a == first_false
        # entries after the first rejection are irrelevant
        if a < k - 1:
            flipped = list(bits)
            flipped[a + 1] = not flipped[a + 1]
            assert SO.leading_ones(np.array([flipped]))[0] == a
    recs, n, draws, _ = _run(top_k=2)
    grow = [sum(int(SO.leading_ones(draws[i])[b]) + 1 for i in range(draws.shape[0]))
            for b in range(draws.shape[1])]
    assert n == [L + 1 + g for L, g in zip((5, 9), grow)]


def test_seed_row_is_causal_softmax_attention():
    """The seed verify of layer 0 attends [0, L_b] with the token's own K/V at
    position L_b: brute force with explicit exponentials over positions."""
    Hq, Hkv, d = 4, 2, 8
    recs, _, _, (w, ctx, e0) = _run(top_k=2, Hq=Hq, Hkv=Hkv, d=d)
    kind, l, r = recs[0]
    assert (kind, l) == ("seed", 0)
    q, kk, vv = SO.project(w[0], e0[:, None, :], Hq, Hkv, d)
    for b, L in enumerate((5, 9)):
        for h in range(Hq):
            kv = h // (Hq // Hkv)
            keys = list(ctx[0][0][b][kv]) + [kk[b, 0, kv]]
            vals = list(ctx[0][1][b][kv]) + [vv[b, 0, kv]]
            logits = [sum(q[b, 0, h, j] * key[j] for j in range(d)) / math.sqrt(d) for key in keys]
            m = max(logits)
            wts = [math.exp(x - m) for x in logits]
            z = sum(wts)
            want = [sum(wts[p] * vals[p][j] for p in range(L + 1)) / z for j in range(d)]
            np.testing.assert_allclose(r["out"][b, 0, h], want, rtol=0, atol=1e-12)
            # captured rows: both rows are the one row, pre-softmax, prefix only
            np.testing.assert_allclose(r["rows"][b, h, 0, :L], logits[:L], rtol=0, atol=1e-12)
            np.testing.assert_allclose(r["rows"][b, h, 1, :L], logits[:L], rtol=0, atol=1e-12)


def test_bf16_rounding_is_round_to_nearest_even():
    x = np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -9, -2.5, 3.0e38])
    got = SO.bf16(x)
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties go to the even mantissa (1.0)
    assert got[0] == 1.0 and got[1] == 1.0
    assert got[2] == 1.0 + 2 * 2.0 ** -7          # 1 + 3*2^-8: halfway, rounds up to even
    assert got[3] == 1.0
    assert got[4] == -2.5
    assert np.isfinite(got[5])


def test_stochastic_rounding_brackets_and_is_unbiased():
    rnd = SO.bf16_stochastic(0)
    x = np.full(20000, 1.0 + 0.3 * 2.0 ** -7)        # 30% of the way from 1 to the next bf16
    y = rnd(x)
    assert set(np.unique(y).tolist()) == {1.0, 1.0 + 2.0 ** -7}
    assert abs(y.mean() - x[0]) < 1e-4   # unbiased: sd of the mean = 2^-7 sqrt(.21/20000) = 2.5e-5
    exact = SO.bf16(np.array([1.5, -3.0, 0.0]))
    np.testing.assert_array_equal(rnd(exact), exact)  # representable values stay put


def test_forcing_a_loop_with_its_own_selections_changes_nothing():
    recs, n, _, _ = _run(top_k=2, lens=(30, 41))
    chosen = iter([r["sets"] for kind, _, r in recs if kind != "draft"])
    w, ctx, e0, draws = _inputs(lens=(30, 41))
    again = []
    n2 = SO.decode_stack(w, ctx, e0, draws, num_q_heads=4, num_kv_heads=2, head_dim=8,
                         prefix_lens=(30, 41), n_drafts=3, top_k=2, n_sink=1, n_recent=2,
                         per_head=False, iterations=3, room=1 + 4 * 4,
                         record=lambda kind, l, r: again.append((kind, l, r)),
                         force_sets=lambda kind, l: next(chosen))
    assert n2 == n
    for (k1, l1, r1), (k2, l2, r2) in zip(recs, again):
        assert (k1, l1) == (k2, l2)
        np.testing.assert_array_equal(r1["out"], r2["out"])
