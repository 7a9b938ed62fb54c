"""Host-side bookkeeping of the decode loop, without a GPU: the accepted
count agrees with the oracle's leading-ones rule on every draw pattern, and
the cache room reserved per sequence covers every position a run writes."""
import itertools

import numpy as np
import torch

from tests.conftest import ensure_lib


def test_accepted_counts_match_oracle_rule():
    ensure_lib()
    from oracle import stack_oracle as SO
    from self_speculative_sparse_vg_gb300.stack import accepted_counts
    k = 5
    pats = np.array(list(itertools.product([False, True], repeat=k)))
    got = accepted_counts(torch.from_numpy(pats)).numpy()
    np.testing.assert_array_equal(got, SO.leading_ones(pats))


def test_room_covers_the_worst_case_run():
    ensure_lib()
    from self_speculative_sparse_vg_gb300.workloads import STACKS, small_stack
    for spec in (STACKS["llama8b_stack32_b4"], small_stack(), small_stack(n_drafts=1)):
        k = spec.n_drafts
        # every draft accepted: the cache grows by k + 1 per iteration after the
        # first token; the last verify writes positions up to n + k
        n = 1
        top = 0
        for _ in range(spec.iterations):
            top = max(top, n + k)
            n += k + 1
        assert top < spec.room
        assert max(spec.prefix_lens) + top < spec.max_prefix + spec.n_drafts + 1
