"""The allocation-free verify entry point against the workspace entry point.

vg_verify_attention_noalloc serves callers that cannot allocate device
memory (a runtime that owns all HBM through its own pool, or a decode loop
that must not call an allocator because cudaMalloc/cudaFree can synchronise
the device).  Its split scratch is a fixed array inside the library, shared
by every call; this test checks that two calls in a row through the C ABI
give the same outputs and captures as the regular entry point with a caller
workspace, within the parity tolerance, and that oversized shapes are
rejected before anything launches."""
import ctypes

import pytest
import torch

from tests import parity_util as P

pytestmark = pytest.mark.gpu


def _require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


@pytest.mark.parametrize("num_splits", [24, 5, 0, 1])  # 24: split scratch in use
def test_noalloc_verify_matches_workspace_entry_point(num_splits):
    _require_gpu()
    from self_speculative_sparse_vg_gb300 import vg
    from self_speculative_sparse_vg_gb300.workloads import make_inputs, small_spec

    spec = small_spec(prefix_lens=(3000, 1777))
    inp = make_inputs(spec)
    dev = torch.device("cuda")
    kv = vg.PagedKV(inp.k_pages.to(dev), inp.v_pages.to(dev), inp.page_table.to(dev))
    q = inp.q_verify.to(dev)
    lens = torch.tensor(spec.prefix_lens, dtype=torch.int32, device=dev)
    B, R, Hq, d = q.shape
    Hkv, Lmax = spec.num_kv_heads, spec.max_prefix
    flag = torch.zeros(1, dtype=torch.int32, device=dev)

    ws = vg.zero_workspace(vg.verify_workspace_bytes(B, R, Hq, Hkv, d, Lmax, num_splits), dev)
    ref_out = torch.zeros(B, R, Hq, d, dtype=torch.bfloat16, device=dev)
    ref_cap = torch.zeros(B, Hkv, Lmax, dtype=torch.float32, device=dev)
    vg.verify_attention(kv, q, lens, Lmax, spec.softmax_scale, ref_out, vg.CAPTURE_GROUP_SUM,
                        ref_cap, num_splits, ws, flag)

    if num_splits == 24:
        assert vg.verify_workspace_bytes(B, R, Hq, Hkv, d, Lmax, num_splits) > 0
    st = kv.struct()
    for _ in range(2):  # two calls in a row share the library's scratch
        out = torch.full((B, R, Hq, d), float("nan"), dtype=torch.bfloat16, device=dev)
        cap = torch.zeros(B, Hkv, Lmax, dtype=torch.float32, device=dev)
        status = vg._lib.vg_verify_attention_noalloc(
            ctypes.byref(st), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(lens.data_ptr()),
            B, R, Hq, Lmax, spec.softmax_scale, ctypes.c_void_p(out.data_ptr()),
            vg.CAPTURE_GROUP_SUM, ctypes.c_void_p(cap.data_ptr()), num_splits,
            ctypes.c_void_p(flag.data_ptr()),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert status == 0, vg.status_string(status)
        torch.cuda.synchronize()
        assert int(flag.item()) == 0
        P.assert_close_out(out.float().cpu().numpy(), ref_out.float().cpu().numpy(), "noalloc out")
        for b, L in enumerate(spec.prefix_lens):
            P.assert_close_capture(cap[b, :, :L].cpu().numpy(), ref_cap[b, :, :L].cpu().numpy(),
                                   "noalloc capture")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    _require_gpu()
    from self_speculative_sparse_vg_gb300 import vg
    limit = vg._lib.vg_verify_noalloc_scratch_bytes()
    assert limit == 16 << 20
    # batch 64, 8 KV heads, 40 rows of 128 at a 128K context with 64 splits
    # needs far more than 16 MiB of split partials
    need = vg.verify_workspace_bytes(64, 8, 40, 8, 128, 131072, 64)
    assert need > limit
    dev = torch.device("cuda")
    pool = torch.zeros(4, 8, 16, 128, dtype=torch.bfloat16, device=dev)
    table = torch.zeros(64, 8200, dtype=torch.int32, device=dev)
    kv = vg.PagedKV(pool, pool, table)
    st = kv.struct()
    dummy = torch.zeros(16, dtype=torch.int32, device=dev)
    p = ctypes.c_void_p(dummy.data_ptr())
    status = vg._lib.vg_verify_attention_noalloc(ctypes.byref(st), p, p, 64, 8, 40, 131072, 0.1,
                                                 p, 0, None, 64, None, None)
    assert status == 3  # VG_ERR_WORKSPACE_TOO_SMALL, nothing launched
