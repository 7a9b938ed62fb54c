"""GPU kernels (through the C ABI) against the float64 oracle."""
from dataclasses import replace

import numpy as np
import pytest
import torch

from tests import parity_util as P

pytestmark = pytest.mark.gpu

vg = pytest.importorskip("self_speculative_sparse_vg_gb300.vg") if torch.cuda.is_available() else None


def _require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def _run(spec, capture_mode=1, per_head=None, num_splits=0):
    from self_speculative_sparse_vg_gb300.step import DecodeStep
    from self_speculative_sparse_vg_gb300.workloads import make_inputs
    inp = make_inputs(spec)
    st = DecodeStep.create(inp, "cuda", capture_mode=capture_mode, per_head=per_head,
                           num_splits=num_splits)
    st.run()
    assert P.flag(st) == 0
    return inp, st


SMALL = dict(
    base={},
    d64=dict(head_dim=64),
    mha=dict(num_q_heads=4, num_kv_heads=4),
    g8=dict(num_q_heads=16, num_kv_heads=2),
    g5=dict(num_q_heads=10, num_kv_heads=2, n_drafts=7),
    k0=dict(n_drafts=0),
    k1=dict(n_drafts=1),
    pages_shuffled=dict(shuffle_pages=True, extra_pages=5),
    short=dict(prefix_lens=(1, 15, 16, 63, 64, 65, 130), batch=7, top_k=8, n_sink=2, n_recent=4),
    budget_all=dict(prefix_lens=(40, 83), top_k=64, n_sink=4, n_recent=16),
    ties=dict(prefix_lens=(700,), batch=1, top_k=33),
    # 24 (sequence, KV head) pairs: the sparse draft's 4-warp CTAs
    many_pairs=dict(batch=3, prefix_lens=(1000, 517, 333), num_q_heads=32, num_kv_heads=8),
    # one long list: a 16-CTA draft cluster merging 15 records into its leader
    long_list=dict(batch=1, prefix_lens=(6000,), num_q_heads=4, num_kv_heads=1, top_k=5500),
    # head_dim 64 with many pairs: the 4-warp draft CTAs at d = 64
    many_pairs_d64=dict(batch=6, prefix_lens=(2000, 1517, 1333, 900, 2100, 1700), head_dim=64,
                        num_q_heads=32, num_kv_heads=8, top_k=512),
)
# drafts without cache slots on a page table longer than the draft kernel
# stages in shared memory (2048 entries): pages looked up entry by entry
NO_SLOTS_EXTRA = dict(
    long_table=dict(batch=1, prefix_lens=(40000,), num_q_heads=4, num_kv_heads=1, top_k=300),
)


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("mode,per_head", [(1, False), (2, False), (1, True), (2, True)])
def test_small_step(name, mode, per_head):
    _require_gpu()
    from self_speculative_sparse_vg_gb300.workloads import small_spec
    spec = small_spec(**SMALL[name])
    inp, st = _run(spec, capture_mode=mode, per_head=per_head)
    P.check_verify(st, inp)
    rows64 = P.oracle_rows(inp)
    P.check_capture(st, inp, rows64)
    P.check_select_end_to_end(st, inp, rows64)
    P.check_slots(st, inp)
    P.check_drafts(st, inp, P.oracle_sets(inp, rows64, per_head))
    P.check_select_synthetic(spec, mode, per_head)
    P.check_drafts_synthetic(st, inp, per_head)


@pytest.mark.parametrize("name", ["base", "d64", "g8", "k0", "pages_shuffled", "short",
                                  "many_pairs", "long_list", "long_table"])
@pytest.mark.parametrize("per_head", [False, True])
def test_draft_without_slots(name, per_head):
    """Drafts on positions alone (no cache slots: the kernel stages the page
    table itself, or looks pages up one by one when the table is long)
    against the oracle, on the GPU's selection and on generator-made index
    lists."""
    _require_gpu()
    from self_speculative_sparse_vg_gb300.step import DecodeStep
    from self_speculative_sparse_vg_gb300.workloads import make_inputs, small_spec
    spec = small_spec(**{**SMALL, **NO_SLOTS_EXTRA}[name])
    inp = make_inputs(spec)
    st = DecodeStep.create(inp, "cuda", per_head=per_head, use_slots=False)
    st.run()
    assert P.flag(st) == 0
    rows64 = P.oracle_rows(inp)
    P.check_select_end_to_end(st, inp, rows64)
    P.check_drafts(st, inp, P.oracle_sets(inp, rows64, per_head))
    P.check_drafts_synthetic(st, inp, per_head)


COLLECT_ALL = ["base", "d64", "mha", "g8", "g5", "k0", "k1", "short", "m96"]
SMALL_EXTRA = dict(m96=dict(num_q_heads=16, num_kv_heads=2, n_drafts=11))  # g*R = 96: 6 row tiles


@pytest.mark.parametrize("name", COLLECT_ALL)
@pytest.mark.parametrize("per_head", [False, True])
def test_small_step_collect_all(name, per_head):
    """Collect-All-Query capture (every verify row summed per KV head) and
    selection on it, against the oracle."""
    _require_gpu()
    from self_speculative_sparse_vg_gb300.workloads import small_spec
    spec = small_spec(**{**SMALL, **SMALL_EXTRA}[name])
    inp, st = _run(spec, capture_mode=3, per_head=per_head)
    P.check_verify(st, inp)
    rows64 = P.oracle_rows(inp)
    P.check_capture(st, inp, rows64)
    P.check_select_end_to_end(st, inp, rows64)
    P.check_drafts(st, inp, P.oracle_sets(inp, rows64, per_head, capture_mode=3))


@pytest.mark.parametrize("name", ["base", "d64", "g8", "g5", "k0", "short", "m96"])
@pytest.mark.parametrize("per_head", [False, True])
def test_small_step_attention_weights(name, per_head):
    """All-rows capture (every row's logits and softmax normaliser) and the
    selection by summed post-softmax weights, against the oracle."""
    _require_gpu()
    from self_speculative_sparse_vg_gb300.workloads import small_spec
    spec = small_spec(**{**SMALL, **SMALL_EXTRA}[name])
    inp, st = _run(spec, capture_mode=4, per_head=per_head)
    P.check_verify(st, inp)
    P.check_capture(st, inp, None)
    P.check_select_end_to_end(st, inp, None)
    P.check_drafts(st, inp, P.oracle_sets(inp, None, per_head, capture_mode=4))


def test_attention_weights_split_invariance():
    """The row normaliser written by the split merge equals the one written
    by a single split, within float32 rounding."""
    _require_gpu()
    from self_speculative_sparse_vg_gb300.workloads import small_spec
    spec = small_spec(prefix_lens=(3000, 1777))
    lses = []
    for ns in (1, 7, 20):
        inp, st = _run(spec, capture_mode=4, num_splits=ns)
        P.check_capture(st, inp, None)
        lses.append(P.split_all_rows(st.capture.cpu().numpy(), spec)[1])
    for x in lses[1:]:
        np.testing.assert_allclose(x, lses[0], rtol=1e-5, atol=1e-5)


def test_ties_select_lower_position():
    """All-equal captured scores: the kept candidates are the lowest positions."""
    _require_gpu()
    from self_speculative_sparse_vg_gb300 import vg as V
    B, Hq, Hkv, L = 1, 8, 2, 3000
    cap = torch.ones(B, Hkv, L, device="cuda")
    cap[0, :, 2000:2010] = 5.0
    lens = torch.tensor([L], dtype=torch.int32, device="cuda")
    idx = torch.full((B, 1, 4 + 16 + 100), -7, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(B, 1, dtype=torch.int32, device="cuda")
    V.select_kv(cap, V.CAPTURE_GROUP_SUM, lens, Hq, Hkv, L, 100, 4, 16, False, idx, cnt)
    torch.cuda.synchronize()
    want = list(range(4)) + list(range(4, 94)) + list(range(2000, 2010)) + list(range(L - 16, L))
    assert idx[0, 0].tolist() == sorted(want)
    assert cnt.item() == 120


def test_split_count_invariance():
    _require_gpu()
    from self_speculative_sparse_vg_gb300.workloads import small_spec
    spec = small_spec(prefix_lens=(3000, 1777))
    outs, caps = [], []
    for ns in (1, 2, 7, 0, 20):  # 20 > 16: merged through the workspace, not a cluster
        inp, st = _run(spec, num_splits=ns)
        outs.append(st.out_verify.float().cpu())
        caps.append(st.capture.cpu())
        P.check_verify(st, inp)
    for o, c in zip(outs[1:], caps[1:]):
        assert (o - outs[0]).abs().max().item() <= 1e-2
        assert torch.equal(c, caps[0])          # logits do not depend on the split


def test_group_sum_equals_ordered_sum_of_rows():
    """Self-consistency of the two capture modes: the per-KV-head sum the
    kernel writes equals, bit for bit, the documented fp32 ordered sum of the
    raw rows it writes in the other mode (computed here with numpy)."""
    _require_gpu()
    from self_speculative_sparse_vg_gb300.workloads import small_spec
    spec = small_spec(num_q_heads=10, num_kv_heads=2)
    _, a = _run(spec, capture_mode=1)
    _, bb = _run(spec, capture_mode=2)
    rows = bb.capture.cpu().numpy()
    g = spec.group
    for b, L in enumerate(spec.prefix_lens):
        for h in range(spec.num_kv_heads):
            acc = rows[b, h * g, 0, :L] + rows[b, h * g, 1, :L]
            for qi in range(1, g):
                acc = acc + (rows[b, h * g + qi, 0, :L] + rows[b, h * g + qi, 1, :L])
            np.testing.assert_array_equal(a.capture.cpu().numpy()[b, h, :L], acc)


def test_poisoned_workspace_and_repeat():
    """Partials must be written before they are read: NaN-filled partials and
    back-to-back calls on one workspace give the same result."""
    _require_gpu()
    from self_speculative_sparse_vg_gb300.step import DecodeStep
    from self_speculative_sparse_vg_gb300.workloads import make_inputs, small_spec
    inp = make_inputs(small_spec(prefix_lens=(2500, 900)))
    st = DecodeStep.create(inp, "cuda", num_splits=20)  # > 16 splits: workspace merge
    st.run()
    ref_v, ref_d = st.out_verify.clone(), st.out_draft.clone()
    assert st.ws_verify.numel() > 1
    st.ws_verify.fill_(0xFF)   # NaN bit patterns in every partial
    P.poison_draft_workspace(st)
    for _ in range(3):
        st.run()
    assert P.flag(st) == 0
    assert torch.equal(st.out_verify, ref_v)
    assert torch.equal(st.out_draft, ref_d)


@pytest.mark.parametrize("kw", [dict(prefix_lens=(3000, 900)),
                                dict(batch=1, prefix_lens=(6000,), num_q_heads=4, num_kv_heads=1,
                                     top_k=5500)], ids=["cluster", "multi_cluster"])
def test_draft_graph_replay_eager_and_empty_list(kw):
    """A captured graph of the draft steps replayed several times and eager
    calls after it are bit-identical to the first eager run, also on a
    NaN-poisoned workspace; an empty attended list gives zeros."""
    _require_gpu()
    from self_speculative_sparse_vg_gb300.step import DecodeStep
    from self_speculative_sparse_vg_gb300.workloads import make_inputs, small_spec
    inp = make_inputs(small_spec(**kw))
    st = DecodeStep.create(inp, "cuda")
    st.run()
    ref = st.out_draft.clone()
    P.poison_draft_workspace(st)   # NaN bit patterns in every chunk record
    k = st.spec.n_drafts
    graph, side = torch.cuda.CUDAGraph(), torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for t in range(1, k + 1):
            st.draft(t, side)  # bind the side stream's arguments outside capture
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=side):
            for t in range(1, k + 1):
                st.draft(t, side)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(3):
        st.out_draft.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(st.out_draft, ref)
    for _ in range(2):
        st.out_draft.fill_(float("nan"))
        for t in range(1, k + 1):
            st.draft(t)
        torch.cuda.synchronize()
        assert torch.equal(st.out_draft, ref)
    assert P.flag(st) == 0
    st.counts.zero_()
    st.cur_len[0].copy_(st.tail_start)
    st.out_draft[0].fill_(float("nan"))
    st.draft(1)
    torch.cuda.synchronize()
    assert P.flag(st) == 0
    assert (st.out_draft[0].float() == 0).all()


@pytest.mark.parametrize("kw", [
    dict(top_k=0, n_sink=4, n_recent=16),                 # no radix pass: sink and recent only
    dict(top_k=50, n_sink=0, n_recent=0),                 # pure top-k
    dict(top_k=1, n_sink=0, n_recent=1),
    # lengths on both sides of the cluster slices (4 CTAs of 1250 positions)
    dict(prefix_lens=(1249, 1250, 1251, 3999, 5000), batch=5, top_k=300, n_sink=3, n_recent=7),
    dict(prefix_lens=(20000,), batch=1, top_k=19000, n_sink=4, n_recent=64),  # nearly all kept
], ids=["top0", "pure_topk", "top1", "slice_edges", "nearly_all"])
@pytest.mark.parametrize("mode,per_head", [(1, False), (1, True), (2, False)])
def test_select_edge_cases(kw, mode, per_head):
    """The selector against the oracle's fp32 mirror on a generator-made
    capture with many exact ties: bit-exact index sets at the edges of its
    parameters and of the cluster's slices."""
    _require_gpu()
    from self_speculative_sparse_vg_gb300.workloads import small_spec
    P.check_select_synthetic(small_spec(**kw), mode, per_head)


def test_device_errors_flag_and_skip():
    """Bad page ids, indices, counts and lengths set the error flag; the
    offending load is skipped (no fault)."""
    _require_gpu()
    from self_speculative_sparse_vg_gb300 import vg as V
    from self_speculative_sparse_vg_gb300.step import DecodeStep
    from self_speculative_sparse_vg_gb300.workloads import make_inputs, small_spec
    inp = make_inputs(small_spec())
    st = DecodeStep.create(inp, "cuda")
    st.kv.page_table[0, 3] = st.kv.k_pages.shape[0] + 5       # out-of-range page id
    st.verify()
    assert P.flag(st) & V.DEVERR_PAGE
    st.error_flag.zero_()
    st.kv.page_table.copy_(inp.page_table.cuda())
    st.run()
    assert P.flag(st) == 0
    good = st.slots[0, 0, 5].item()
    st.slots[0, 0, 5] = (good & ~15) | ((good + 1) & 15)      # slot of another offset in its page
    st.draft(1)
    assert P.flag(st) == V.DEVERR_INDEX
    st.error_flag.zero_()
    st.slots[0, 0, 5] = (st.kv.k_pages.shape[0] + 3) * 16 + (good & 15)  # page outside the pool
    st.draft(1)
    assert P.flag(st) == V.DEVERR_PAGE
    st.error_flag.zero_()
    st.slots[0, 0, 5] = good
    st.draft(1)
    assert P.flag(st) == 0
    st.indices[0, 0, 0] = int(st.prefix_lens[0]) + 3          # index beyond the prefix
    st.draft(1)
    assert P.flag(st) & V.DEVERR_INDEX
    st.error_flag.zero_()
    st.counts[1, 0] = st.indices.shape[-1] + 1                # count above cap
    st.draft(1)
    assert P.flag(st) & V.DEVERR_COUNT
    st.error_flag.zero_()
    st.prefix_lens[1] = st.spec.max_prefix + 1               # length above the host bound
    st.verify()
    st.select()
    assert P.flag(st) & V.DEVERR_LENGTH


FULL = ["tiny_d64_2k", "llama8b_32k", "llama8b_b8_16k_64k", "qwen14b_128k"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload(name):
    """Full-size workloads in the launch configuration the benchmark uses:
    sampled (sequence, KV head) pairs for attention, the selector bit-exact
    against the fp32 mirror on a synthetic capture of the workload's shape,
    end-to-end selection within the gap rule."""
    _require_gpu()
    from self_speculative_sparse_vg_gb300.workloads import WORKLOADS
    spec = WORKLOADS[name]
    modes = [(1, False), (2, True), (3, False)] if spec.batch > 1 else [(1, False), (3, True)]
    for mode, per_head in modes:
        inp, st = _run(spec, capture_mode=mode, per_head=per_head)
        if name == "tiny_d64_2k":
            pairs = None
        else:  # every KV head of the first and of the last sequence
            pairs = sorted({(b, h) for b in (0, spec.batch - 1) for h in range(spec.num_kv_heads)})
        P.check_verify(st, inp, pairs)
        rows64 = P.oracle_rows(inp)
        P.check_capture(st, inp, rows64)
        P.check_select_end_to_end(st, inp, rows64)
        P.check_slots(st, inp)
        osets = P.oracle_sets(inp, rows64, per_head, capture_mode=mode)
        P.check_drafts(st, inp, osets, pairs=pairs, steps=[1, spec.n_drafts])
        if name == "tiny_d64_2k":
            assert set(inp.planted[0].tolist()) <= set(P.gpu_sets(st)[0][0].tolist())
        if mode != 3:  # Collect-All feeds the selector the same layout as mode 1
            P.check_select_synthetic(spec, mode, per_head)
        P.check_drafts_synthetic(st, inp, per_head, pairs=pairs, steps=[1, spec.n_drafts])
        del st
        torch.cuda.empty_cache()


# More units (split x KV head x sequence) than SMs: persistent verify CTAs
# each walk several units; ragged lengths give short last splits and
# sequences with a single tile; M = g * R covers the 4-, 2- and 1-copy
# layouts (96 rows: one softmax warp idle).
PERSIST = dict(
    ragged=dict(batch=4, prefix_lens=(3000, 9000, 1, 6001), num_q_heads=32, num_kv_heads=8,
                top_k=200),
    r8=dict(batch=3, prefix_lens=(4096, 4100, 2222), num_q_heads=32, num_kv_heads=8,
            n_drafts=7),
    m48=dict(batch=4, prefix_lens=(9000, 5000, 7777, 100), num_q_heads=16, num_kv_heads=2,
             n_drafts=5),
    m96=dict(batch=4, prefix_lens=(9000, 5000, 7777, 100), num_q_heads=16, num_kv_heads=2,
             n_drafts=11),
)


@pytest.mark.parametrize("name", list(PERSIST))
@pytest.mark.parametrize("mode", [1, 2, 3, 4])
def test_persistent_verify(name, mode):
    _require_gpu()
    from self_speculative_sparse_vg_gb300.workloads import small_spec
    spec = small_spec(**PERSIST[name])
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles = -(-(spec.max_prefix + spec.n_rows) // 128)
    ran = 0
    for ns in (40, 16, 71):  # 71: one-tile units
        tps = -(-tiles // min(ns, tiles))
        splits = -(-tiles // tps)
        if spec.batch * spec.num_kv_heads * splits <= sms:
            continue  # not the persistent path
        ran += 1
        inp, st = _run(spec, capture_mode=mode, num_splits=ns)
        P.check_verify(st, inp)
        rows64 = P.oracle_rows(inp) if mode != 4 else None
        P.check_capture(st, inp, rows64)
        P.check_select_end_to_end(st, inp, rows64)
    assert ran >= 2


def test_persistent_verify_skipped_sequence_and_repeat():
    """A sequence whose length exceeds its bound is flagged and skipped by
    the persistent CTAs; the others are unaffected, and a repeated call on a
    NaN-poisoned workspace gives the same bits."""
    _require_gpu()
    from self_speculative_sparse_vg_gb300 import vg as V
    from self_speculative_sparse_vg_gb300.workloads import small_spec
    spec = small_spec(**PERSIST["ragged"])
    inp, st = _run(spec, num_splits=40)
    ref = st.out_verify.clone()
    st.ws_verify.fill_(0xFF)
    st.verify()
    assert P.flag(st) == 0
    assert torch.equal(st.out_verify, ref)
    st.prefix_lens[2] = spec.max_prefix + 1
    st.out_verify.fill_(0)
    st.verify()
    assert P.flag(st) & V.DEVERR_LENGTH
    keep = [0, 1, 3]
    assert torch.equal(st.out_verify[keep], ref[keep])
