"""Sparse verification (SSV exact merged schedule) through the C ABI against
the float64 oracle: every verify row attends its own 16-position prefix
blocks plus the verify block causally; the kernel streams the union of the
rows' blocks once per KV head."""
import pytest
import torch

from tests import parity_util as P

pytestmark = pytest.mark.gpu


def _require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def _run(spec, frac, seed=3, num_splits=0, blocks=None):
    from self_speculative_sparse_vg_gb300 import vg
    from self_speculative_sparse_vg_gb300.workloads import make_block_selection, make_inputs
    inp = make_inputs(spec)
    dev = torch.device("cuda")
    kv = vg.PagedKV(inp.k_pages.to(dev), inp.v_pages.to(dev), inp.page_table.to(dev))
    if blocks is None:
        blocks, counts = make_block_selection(spec, frac, seed)
    else:
        blocks, counts = blocks
    q = inp.q_verify.to(dev)
    lens = torch.tensor(spec.prefix_lens, dtype=torch.int32, device=dev)
    out = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device=dev)
    flag = torch.zeros(1, dtype=torch.int32, device=dev)
    vg.sparse_verify_attention(kv, q, lens, spec.max_prefix, spec.softmax_scale, blocks.to(dev),
                               counts.to(dev), out, num_splits=num_splits, error_flag=flag)
    torch.cuda.synchronize()
    return inp, out.float().cpu().numpy(), int(flag.item()), blocks, counts


def _oracle(inp, blocks, counts, pairs=None):
    from oracle import vg_oracle as O
    s = inp.spec
    sel = [[blocks[b, i, :counts[b, i]].tolist() for i in range(s.n_rows)] for b in range(s.batch)]
    q, k, v = P.dense64(inp)
    if pairs is None:
        return O.sparse_verify_attention(q, k, v, s.prefix_lens, sel, s.softmax_scale), None
    res = {}
    g = s.group
    for b, h in pairs:
        qs, ks, vs = P.sub_problem(q, k, v, b, h, g)
        res[(b, h)] = O.sparse_verify_attention(qs, ks, vs, [s.prefix_lens[b]], [sel[b]],
                                                s.softmax_scale)[0]
    return None, res


CASES = dict(
    base={}, d64=dict(head_dim=64), g8=dict(num_q_heads=16, num_kv_heads=2),
    g5=dict(num_q_heads=10, num_kv_heads=2, n_drafts=7),
    m96=dict(num_q_heads=16, num_kv_heads=2, n_drafts=11), k0=dict(n_drafts=0),
    short=dict(prefix_lens=(1, 15, 16, 63, 64, 65, 130), batch=7),
    pages_shuffled=dict(shuffle_pages=True, extra_pages=5),
)


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("frac", [0.0, 0.1, 0.5, 1.0])
def test_sparse_verify_matches_oracle(name, frac):
    _require_gpu()
    from self_speculative_sparse_vg_gb300.workloads import small_spec
    spec = small_spec(**CASES[name])
    inp, got, flag, blocks, counts = _run(spec, frac)
    assert flag == 0
    ref, _ = _oracle(inp, blocks, counts)
    P.assert_close_out(got, ref, f"sparse verify {name} frac={frac}")


@pytest.mark.parametrize("num_splits", [1, 3, 20])
def test_sparse_verify_split_counts(num_splits):
    _require_gpu()
    from self_speculative_sparse_vg_gb300.workloads import small_spec
    spec = small_spec(prefix_lens=(3000, 1777))
    inp, got, flag, blocks, counts = _run(spec, 0.3, num_splits=num_splits)
    assert flag == 0
    ref, _ = _oracle(inp, blocks, counts)
    P.assert_close_out(got, ref, f"sparse verify splits={num_splits}")


def test_sparse_verify_flags_bad_blocks_and_counts():
    _require_gpu()
    from self_speculative_sparse_vg_gb300 import vg as V
    from self_speculative_sparse_vg_gb300.workloads import make_block_selection, small_spec
    spec = small_spec()
    blocks, counts = make_block_selection(spec, 0.2, 5)
    bad = blocks.clone()
    bad[0, 1, 0] = (spec.prefix_lens[0] + 15) // 16 + 3       # past the prefix
    _, _, flag, _, _ = _run(spec, 0.2, blocks=(bad, counts))
    assert flag & V.DEVERR_INDEX
    badc = counts.clone()
    badc[1, 0] = blocks.shape[-1] + 1                         # above max_blocks
    _, _, flag, _, _ = _run(spec, 0.2, blocks=(blocks, badc))
    assert flag & V.DEVERR_COUNT


@pytest.mark.parametrize("name", ["llama8b_32k", "qwen14b_128k"])
def test_sparse_verify_full_size(name):
    """About 7 % of the blocks per row, the rows sharing three quarters of
    them; sampled (sequence, KV head) pairs against the oracle."""
    _require_gpu()
    from self_speculative_sparse_vg_gb300.workloads import WORKLOADS
    spec = WORKLOADS[name]
    inp, got, flag, blocks, counts = _run(spec, 0.07)
    assert flag == 0
    pairs = [(0, 0), (spec.batch - 1, spec.num_kv_heads - 1)]
    _, res = _oracle(inp, blocks, counts, pairs)
    g = spec.group
    for (b, h), ref in res.items():
        P.assert_close_out(got[b, :, h * g:(h + 1) * g], ref, f"{name} b={b} h={h}")
