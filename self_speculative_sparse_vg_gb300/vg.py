"""Thin Python binding of libvg.so (the C ABI in include/vg.h).

Argument marshalling only: tensors in, device pointers and sizes out, the
current torch stream passed through.  Every step of the hot path runs in the
library's CUDA kernels; if the library is missing this module raises on
import -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libvg.so")

CAPTURE_NONE = 0
CAPTURE_GROUP_SUM = 1
CAPTURE_ROWS = 2
CAPTURE_ALL_SUM = 3
CAPTURE_ALL_ROWS = 4

DEVERR_PAGE = 1
DEVERR_INDEX = 2
DEVERR_COUNT = 4
DEVERR_TIMEOUT = 8
DEVERR_LENGTH = 16

EXPORTED = (
    "vg_verify_workspace_bytes", "vg_verify_attention",
    "vg_select_workspace_bytes", "vg_select_launches", "vg_select_kv", "vg_select_kv_weights",
    "vg_sparse_draft_workspace_bytes", "vg_sparse_draft_attention",
    "vg_status_string", "vg_version",
    "vg_verify_noalloc_scratch_bytes", "vg_verify_attention_noalloc",
    "vg_sparse_verify_workspace_bytes", "vg_sparse_verify_attention",
    "vg_set_wait_limit_ns",
)


class VGError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")


class PagedKVStruct(ctypes.Structure):
    _fields_ = [("k_pages", ctypes.c_void_p), ("v_pages", ctypes.c_void_p),
                ("page_table", ctypes.c_void_p), ("num_pages", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("max_pages_per_seq", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"{_LIB_PATH} is not built; run `python -c \"import __graft_entry__ as g; "
                          f"g.build()\"` (needs nvcc with sm_103a support)")
    lib = ctypes.CDLL(_LIB_PATH)
    vp, i32, sz, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
    kvp = ctypes.POINTER(PagedKVStruct)
    sig = {
        "vg_verify_workspace_bytes": (sz, [i32, i32, i32, i32, i32, i32, i32]),
        "vg_verify_attention": (i32, [kvp, vp, vp, i32, i32, i32, i32, f32, vp, i32, vp, i32,
                                      vp, sz, vp, vp]),
        "vg_select_workspace_bytes": (sz, [i32, i32, i32, i32]),
        "vg_select_launches": (i32, [i32, i32, i32, i32, i32]),
        "vg_select_kv_weights": (i32, [vp, i32, vp, i32, i32, i32, i32, i32, i32, i32, i32, vp,
                                       vp, i32, kvp, vp, vp, sz, vp, vp]),
        "vg_select_kv": (i32, [vp, i32, vp, i32, i32, i32, i32, i32, i32, i32, i32, vp, vp, i32,
                               kvp, vp, vp, sz, vp, vp]),
        "vg_sparse_draft_workspace_bytes": (sz, [i32, i32, i32, i32, i32, i32]),
        "vg_sparse_draft_attention": (i32, [kvp, vp, vp, vp, vp, i32, i32, vp, vp, i32, i32, i32,
                                            f32, vp, vp, sz, vp, vp]),
        "vg_verify_noalloc_scratch_bytes": (sz, []),
        "vg_verify_attention_noalloc": (i32, [kvp, vp, vp, i32, i32, i32, i32, f32, vp, i32, vp,
                                              i32, vp, vp]),
        "vg_sparse_verify_workspace_bytes": (sz, [i32, i32, i32, i32, i32, i32, i32, i32]),
        "vg_sparse_verify_attention": (i32, [kvp, vp, vp, i32, i32, i32, i32, f32, vp, vp, i32, vp,
                                             i32, vp, sz, vp, vp]),
        "vg_set_wait_limit_ns": (i32, [ctypes.c_uint64]),
        "vg_status_string": (ctypes.c_char_p, [i32]),
        "vg_version": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def set_wait_limit_ns(limit_ns: int) -> None:
    """vg_set_wait_limit_ns: waits longer than limit_ns report
    DEVERR_TIMEOUT (and go on, up to 1 s); 0 restores the default."""
    _check("vg_set_wait_limit_ns", _lib.vg_set_wait_limit_ns(int(limit_ns)))


def status_string(s: int) -> str:
    return _lib.vg_status_string(int(s)).decode()


def version() -> str:
    return _lib.vg_version().decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn, status):
    if status != 0:
        raise VGError(fn, status)


@dataclass
class PagedKV:
    """Paged bf16 KV cache: pools [P][Hkv][16][d], page table [B][max_pages]."""
    k_pages: torch.Tensor
    v_pages: torch.Tensor
    page_table: torch.Tensor

    def __post_init__(self):
        assert self.k_pages.dtype == torch.bfloat16 and self.v_pages.dtype == torch.bfloat16
        assert self.k_pages.shape == self.v_pages.shape and self.k_pages.dim() == 4
        assert self.page_table.dtype == torch.int32 and self.page_table.dim() == 2
        assert self.k_pages.is_contiguous() and self.v_pages.is_contiguous()
        assert self.page_table.is_contiguous()

    @property
    def num_kv_heads(self):
        return self.k_pages.shape[1]

    @property
    def head_dim(self):
        return self.k_pages.shape[3]

    def struct(self) -> PagedKVStruct:
        P, H, S, D = self.k_pages.shape
        return PagedKVStruct(self.k_pages.data_ptr(), self.v_pages.data_ptr(),
                             self.page_table.data_ptr(), P, S, self.page_table.shape[1], H, D)


# --------------------------------------------------------------------- verify
def verify_workspace_bytes(batch, n_rows, num_q_heads, num_kv_heads, head_dim, max_prefix,
                           num_splits=0) -> int:
    return int(_lib.vg_verify_workspace_bytes(batch, n_rows, num_q_heads, num_kv_heads, head_dim,
                                              max_prefix, num_splits))


def verify_attention(kv: PagedKV, q, prefix_lens, max_prefix, softmax_scale, out,
                     capture_mode=CAPTURE_GROUP_SUM, capture=None, num_splits=0, workspace=None,
                     error_flag=None, stream=None):
    """vg_verify_attention.  q [B][R][Hq][d] bf16, prefix_lens int32 [B]."""
    B, R, Hq, _ = q.shape
    st = kv.struct()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    s = _lib.vg_verify_attention(ctypes.byref(st), _ptr(q), _ptr(prefix_lens), B, R, Hq,
                                 int(max_prefix), float(softmax_scale), _ptr(out),
                                 int(capture_mode), _ptr(capture), int(num_splits),
                                 _ptr(workspace), ws_bytes, _ptr(error_flag), _stream(stream))
    _check("vg_verify_attention", s)
    return out


def verify_attention_noalloc(kv: PagedKV, q, prefix_lens, max_prefix, softmax_scale, out,
                             capture_mode=CAPTURE_GROUP_SUM, capture=None, num_splits=0,
                             error_flag=None, stream=None):
    """vg_verify_attention_noalloc: same result, scratch in the library's
    fixed device array instead of a caller workspace."""
    B, R, Hq, _ = q.shape
    st = kv.struct()
    s = _lib.vg_verify_attention_noalloc(ctypes.byref(st), _ptr(q), _ptr(prefix_lens), B, R, Hq,
                                         int(max_prefix), float(softmax_scale), _ptr(out),
                                         int(capture_mode), _ptr(capture), int(num_splits),
                                         _ptr(error_flag), _stream(stream))
    _check("vg_verify_attention_noalloc", s)
    return out


def sparse_verify_workspace_bytes(batch, n_rows, num_q_heads, num_kv_heads, head_dim, max_prefix,
                                  max_blocks, num_splits=0) -> int:
    return int(_lib.vg_sparse_verify_workspace_bytes(batch, n_rows, num_q_heads, num_kv_heads,
                                                     head_dim, max_prefix, max_blocks, num_splits))


def sparse_verify_attention(kv: PagedKV, q, prefix_lens, max_prefix, softmax_scale, blocks,
                            block_counts, out, num_splits=0, workspace=None, error_flag=None,
                            stream=None):
    """vg_sparse_verify_attention.  blocks int32 [B][R][max_blocks] (16-position
    prefix blocks per verify row), block_counts int32 [B][R]."""
    B, R, Hq, d = q.shape
    max_blocks = blocks.shape[-1]
    if workspace is None:
        workspace = zero_workspace(sparse_verify_workspace_bytes(
            B, R, Hq, kv.num_kv_heads, d, max_prefix, max_blocks, num_splits), q.device)
    st = kv.struct()
    s = _lib.vg_sparse_verify_attention(ctypes.byref(st), _ptr(q), _ptr(prefix_lens), B, R, Hq,
                                        int(max_prefix), float(softmax_scale), _ptr(blocks),
                                        _ptr(block_counts), int(max_blocks), _ptr(out),
                                        int(num_splits), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(),
                                        _ptr(error_flag), _stream(stream))
    _check("vg_sparse_verify_attention", s)
    return out


# --------------------------------------------------------------------- select
def select_workspace_bytes(batch, num_kv_heads, max_prefix, per_head) -> int:
    return int(_lib.vg_select_workspace_bytes(batch, num_kv_heads, max_prefix, int(bool(per_head))))


def select_launches(capture_mode, batch, num_kv_heads, max_prefix, per_head) -> int:
    """Kernels one selection call launches for this shape on the current
    device (1 or 2; 0 for an unsupported shape)."""
    return int(_lib.vg_select_launches(int(capture_mode), batch, num_kv_heads, max_prefix,
                                       int(bool(per_head))))


def _kv_arg(kv, slots):
    if slots is None:
        return None, None
    assert kv is not None, "slots need the paged cache whose page table they translate"
    return kv.struct(), slots


def select_kv(capture, capture_mode, prefix_lens, num_q_heads, num_kv_heads, max_prefix, top_k,
              n_sink, n_recent, per_head, indices, counts, error_flag=None, stream=None,
              workspace=None, kv=None, slots=None):
    """vg_select_kv.  indices int32 [B][rows][cap], counts int32 [B][rows];
    slots (optional, with kv) int32 like indices: the cache slots of the kept
    positions.  workspace: uint8 device tensor of select_workspace_bytes()
    (allocated here when not given)."""
    B = prefix_lens.shape[0]
    cap = indices.shape[-1]
    if workspace is None:
        workspace = zero_workspace(select_workspace_bytes(B, num_kv_heads, max_prefix, per_head),
                                   indices.device)
    st, slots = _kv_arg(kv, slots)
    s = _lib.vg_select_kv(_ptr(capture), int(capture_mode), _ptr(prefix_lens), B, num_q_heads,
                          num_kv_heads, int(max_prefix), int(top_k), int(n_sink), int(n_recent),
                          int(bool(per_head)), _ptr(indices), _ptr(counts), cap,
                          None if st is None else ctypes.byref(st), _ptr(slots), _ptr(workspace),
                          workspace.numel(), _ptr(error_flag), _stream(stream))
    _check("vg_select_kv", s)
    return indices, counts


def all_rows_capture_floats(batch, num_q_heads, n_rows, max_prefix) -> int:
    """Float count of a VG_CAPTURE_ALL_ROWS capture: logits, then row lse."""
    return batch * num_q_heads * n_rows * (max_prefix + 1)


def select_kv_weights(capture, n_rows, prefix_lens, num_q_heads, num_kv_heads, max_prefix,
                      top_k, n_sink, n_recent, per_head, indices, counts, error_flag=None,
                      stream=None, workspace=None, kv=None, slots=None):
    """vg_select_kv_weights: selection by the post-softmax weights of the
    n_rows captured rows (capture from VG_CAPTURE_ALL_ROWS)."""
    B = prefix_lens.shape[0]
    cap = indices.shape[-1]
    if workspace is None:
        workspace = zero_workspace(select_workspace_bytes(B, num_kv_heads, max_prefix, per_head),
                                   indices.device)
    st, slots = _kv_arg(kv, slots)
    s = _lib.vg_select_kv_weights(_ptr(capture), int(n_rows), _ptr(prefix_lens), B, num_q_heads,
                                  num_kv_heads, int(max_prefix), int(top_k), int(n_sink),
                                  int(n_recent), int(bool(per_head)), _ptr(indices), _ptr(counts),
                                  cap, None if st is None else ctypes.byref(st), _ptr(slots),
                                  _ptr(workspace), workspace.numel(), _ptr(error_flag),
                                  _stream(stream))
    _check("vg_select_kv_weights", s)
    return indices, counts


# ---------------------------------------------------------------- sparse draft
def sparse_draft_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, cap, max_tail) -> int:
    return int(_lib.vg_sparse_draft_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim,
                                                    cap, max_tail))


def sparse_draft_attention(kv: PagedKV, q, indices, counts, per_head, tail_start, cur_len,
                           max_tail, softmax_scale, out, workspace=None, error_flag=None,
                           stream=None, slots=None):
    """vg_sparse_draft_attention.  q [B][Hq][d] bf16; slots (optional) as
    written by select_kv beside the indices.  No workspace is needed (the
    argument is accepted and ignored)."""
    B, Hq, _ = q.shape
    st = kv.struct()
    cap = indices.shape[-1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    s = _lib.vg_sparse_draft_attention(ctypes.byref(st), _ptr(q), _ptr(indices), _ptr(slots),
                                       _ptr(counts),
                                       int(bool(per_head)), cap, _ptr(tail_start), _ptr(cur_len),
                                       B, Hq, int(max_tail), float(softmax_scale), _ptr(out),
                                       _ptr(workspace), ws_bytes, _ptr(error_flag),
                                       _stream(stream))
    _check("vg_sparse_draft_attention", s)
    return out


def zero_workspace(nbytes: int, device) -> torch.Tensor:
    """A zero-filled byte workspace of at least one byte (zeros only keep a
    fresh buffer free of stale bytes: every workspace is written before it
    is read)."""
    return torch.zeros(max(int(nbytes), 1), dtype=torch.uint8, device=device)
