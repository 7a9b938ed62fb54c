"""Failure detection without a GPU fault: a short wait bound makes the
kernels report VG_DEVERR_TIMEOUT, and the calls still complete with the
same results (a reported wait goes on waiting, so nothing is abandoned in
flight).  The bound is restored afterwards and a clean run reports
nothing."""
import pytest
import torch

from tests import parity_util as P

pytestmark = pytest.mark.gpu


def _require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


@pytest.mark.parametrize("use_slots", [True, False])
def test_short_wait_bound_reports_and_completes(use_slots):
    _require_gpu()
    from self_speculative_sparse_vg_gb300 import vg
    from self_speculative_sparse_vg_gb300.step import DecodeStep
    from self_speculative_sparse_vg_gb300.workloads import make_inputs, small_spec
    # large enough that the draft's gathers wait microseconds on DRAM
    inp = make_inputs(small_spec(prefix_lens=(30000, 20000), num_q_heads=32, num_kv_heads=8,
                                 top_k=2048, n_sink=4, n_recent=64, n_drafts=5))
    st = DecodeStep.create(inp, "cuda", use_slots=use_slots)
    st.run()
    assert P.flag(st) == 0
    ref_v, ref_d = st.out_verify.clone(), st.out_draft.clone()
    ref_i, ref_c = st.indices.clone(), st.counts.clone()
    vg.set_wait_limit_ns(1)
    try:
        st.out_verify.fill_(float("nan"))
        st.verify()
        assert P.flag(st) == vg.DEVERR_TIMEOUT      # reported, nothing else
        assert torch.equal(st.out_verify, ref_v)   # and the call completed
        st.error_flag.zero_()
        st.select()
        assert P.flag(st) & ~vg.DEVERR_TIMEOUT == 0
        assert torch.equal(st.indices, ref_i) and torch.equal(st.counts, ref_c)
        st.error_flag.zero_()
        st.out_draft.fill_(float("nan"))
        # rows from DRAM, not L2: the gathers wait long enough to pass the
        # bound (the device timer ticks every few hundred nanoseconds)
        l2 = torch.cuda.get_device_properties(0).L2_cache_size
        cold = torch.ones(int(1.5 * l2) // 4, device="cuda")
        for t in range(1, st.spec.n_drafts + 1):
            cold.sum()
            st.draft(t)
        assert P.flag(st) == vg.DEVERR_TIMEOUT
        assert torch.equal(st.out_draft, ref_d)
    finally:
        vg.set_wait_limit_ns(0)
    st.error_flag.zero_()
    st.run()
    assert P.flag(st) == 0
    assert torch.equal(st.out_verify, ref_v) and torch.equal(st.out_draft, ref_d)
