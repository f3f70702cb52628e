"""Exact tiled attention on GB300 (sm_103a) — Python binding of the C ABI.

The functions ``fa_fwd``, ``fa_bwd`` (and its steps ``fa_bwd_preprocess``,
``fa_bwd_dkdv``, ``fa_bwd_dq``), ``fa_decode``, ``fa_bwd_workspace_bytes``,
``fa_decode_workspace_bytes``, ``fa_get_last_device_error``,
``fa_set_wait_timeout_ns``, ``fa_status_string`` and ``fa_version`` carry the
names and arguments of ``include/fa.h`` and only marshal arguments: every step
of the computation runs in the CUDA kernels of ``libfa_gb300.so``.  PyTorch
supplies device memory (``data_ptr``) and the stream.  ``forward``,
``backward`` and ``decode`` are conveniences that allocate the outputs and the
workspace with torch and then call the same entry points.

There is no fallback: if the shared library is missing, or a call returns an
error status, a ``FAError`` is raised.
"""
import ctypes
import math
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa_gb300.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "fa.h")

FA_OK = 0
FA_ERR_INVALID_ARG = -1
FA_ERR_UNSUPPORTED = -2
FA_ERR_ALIGNMENT = -3
FA_ERR_WORKSPACE = -4
FA_ERR_CUDA = -5
FA_ERR_TIMEOUT = -6

_lib = None

_NAMES = {FA_OK: "FA_OK", FA_ERR_INVALID_ARG: "FA_ERR_INVALID_ARG",
          FA_ERR_UNSUPPORTED: "FA_ERR_UNSUPPORTED", FA_ERR_ALIGNMENT: "FA_ERR_ALIGNMENT",
          FA_ERR_WORKSPACE: "FA_ERR_WORKSPACE", FA_ERR_CUDA: "FA_ERR_CUDA",
          FA_ERR_TIMEOUT: "FA_ERR_TIMEOUT"}


class FAError(RuntimeError):
    """A C-ABI call returned a status other than FA_OK (or the library is missing)."""

    def __init__(self, status, what):
        self.status = status
        super().__init__("%s failed: %s (%d)" % (what, _NAMES.get(status, "?"), status))


def build(force=False):
    """Compile libfa_gb300.so in-tree (nvcc, sm_103a) and return its path."""
    from . import _build
    return _build.build(force=force)


def load():
    """Load the shared library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise FAError(FA_ERR_CUDA, "loading %s (not built; call build())" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    lib.fa_fwd.restype = i
    lib.fa_bwd_workspace_bytes.argtypes = [i, i, i, i, i]
    lib.fa_bwd_workspace_bytes.restype = sz
    lib.fa_bwd.argtypes = [vp] * 9 + [i, i, i, i, i, f, i, vp, sz, vp]
    lib.fa_bwd.restype = i
    lib.fa_bwd_fused_workspace_bytes.argtypes = [i, i, i, i, i]
    lib.fa_bwd_fused_workspace_bytes.restype = sz
    lib.fa_bwd_fused.argtypes = [vp] * 9 + [i, i, i, i, i, f, i, vp, sz, vp]
    lib.fa_bwd_fused.restype = i
    lib.fa_bwd_preprocess.argtypes = [vp, vp, vp, i, i, i, i, vp]
    lib.fa_bwd_preprocess.restype = i
    lib.fa_bwd_dkdv.argtypes = [vp] * 8 + [i, i, i, i, i, f, i, vp]
    lib.fa_bwd_dkdv.restype = i
    lib.fa_bwd_dkdv_pair.argtypes = [vp] * 8 + [i, i, i, i, i, f, i, vp]
    lib.fa_bwd_dkdv_pair.restype = i
    lib.fa_bwd_dq.argtypes = [vp] * 7 + [i, i, i, i, i, f, i, vp]
    lib.fa_bwd_dq.restype = i
    lib.fa_decode_workspace_bytes.argtypes = [i, i, i, i, i]
    lib.fa_decode_workspace_bytes.restype = sz
    lib.fa_decode.argtypes = [vp] * 5 + [i, i, i, i, f, i, vp, sz, vp]
    lib.fa_decode.restype = i
    lib.fa_get_last_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_int)]
    lib.fa_get_last_device_error.restype = i
    lib.fa_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
    lib.fa_set_wait_timeout_ns.restype = ctypes.c_uint64
    lib.fa_status_string.argtypes = [i]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_version.argtypes = []
    lib.fa_version.restype = i
    lib.fa_fwd_tile_rows.argtypes = [i] * 6
    lib.fa_fwd_tile_rows.restype = i
    lib.fa_work_schedule.argtypes = [i, i, i, i, ctypes.POINTER(ctypes.c_int)]
    lib.fa_work_schedule.restype = i
    _lib = lib
    return lib


def declared_symbols():
    """Names of the functions declared in include/fa.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", text)))


# ------------------------------------------------------------------ raw entry points
def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _raise(status, what):
    if status != FA_OK:
        raise FAError(status, what)


def fa_status_string(status):
    try:
        return load().fa_status_string(int(status)).decode()
    except FAError:
        return "status %d" % status


def fa_version():
    return load().fa_version()


def fa_set_wait_timeout_ns(ns):
    return int(load().fa_set_wait_timeout_ns(int(ns)))


def fa_get_last_device_error(stream=None):
    """Synchronise the stream; return (status, [code, site, block, aux]) and clear the word."""
    detail = (ctypes.c_int * 4)()
    st = load().fa_get_last_device_error(_stream(stream), detail)
    return st, list(detail)


def fa_decode_paged_workspace_bytes(B, Hq, d, num_splits):
    fn = load().fa_decode_paged_workspace_bytes
    fn.argtypes = [ctypes.c_int] * 4
    fn.restype = ctypes.c_size_t
    return int(fn(B, Hq, d, num_splits))


def fa_decode_paged(q, k_pages, v_pages, block_table, seq_lens, o, lse, B, Hq, Hkv, page_size,
                    max_pages, num_pages, d, scale, num_splits, workspace, workspace_bytes, stream=None):
    fn = load().fa_decode_paged
    if fn.argtypes is None:
        vp, i = ctypes.c_void_p, ctypes.c_int
        fn.argtypes = [vp] * 7 + [i] * 7 + [ctypes.c_float, i, vp, ctypes.c_size_t, vp]
        fn.restype = ctypes.c_int
    _raise(fn(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), _ptr(seq_lens), _ptr(o), _ptr(lse),
              B, Hq, Hkv, page_size, max_pages, num_pages, d, float(scale), int(num_splits),
              _ptr(workspace), int(workspace_bytes), _stream(stream)), "fa_decode_paged")


def decode_paged(q, k_pages, v_pages, block_table, seq_lens, scale=None, num_splits=0, stream=None):
    """O [B,Hq,d] bf16 and LSE [B,Hq] fp32 against a paged cache (int32 table and lengths on the device).
    num_splits <= 0: the library's choice."""
    B, Hq, d = q.shape
    num_pages, Hkv, page_size = k_pages.shape[:3]
    max_pages = block_table.shape[1]
    for t, n in ((q, "q"), (k_pages, "k_pages"), (v_pages, "v_pages")):
        if not (t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()):
            raise ValueError("%s must be a contiguous bf16 CUDA tensor" % n)
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise ValueError("block_table and seq_lens must be int32")
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    ws = torch.empty(fa_decode_paged_workspace_bytes(B, Hq, d, num_splits), dtype=torch.uint8, device=q.device)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    fa_decode_paged(q, k_pages, v_pages, block_table, seq_lens, o, lse, B, Hq, Hkv, page_size, max_pages,
                    num_pages, d, scale, num_splits, ws, ws.numel(), stream)
    return o, lse


def fa_fwd_window(q, k, v, o, lse, B, H, Nq, Nk, d, scale, window, stream=None):
    fn = load().fa_fwd_window
    if fn.argtypes is None:
        vp, i = ctypes.c_void_p, ctypes.c_int
        fn.argtypes = [vp] * 5 + [i] * 5 + [ctypes.c_float, i, vp]
        fn.restype = i
    _raise(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nk, d, float(scale), int(window),
              _stream(stream)), "fa_fwd_window")


def fa_bwd_window(q, k, v, o, lse, dO, dq, dk, dv, B, H, Nq, Nk, d, scale, window, workspace,
                  workspace_bytes, stream=None):
    fn = load().fa_bwd_window
    if fn.argtypes is None:
        vp, i = ctypes.c_void_p, ctypes.c_int
        fn.argtypes = [vp] * 9 + [i] * 5 + [ctypes.c_float, i, vp, ctypes.c_size_t, vp]
        fn.restype = i
    _raise(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv), B, H, Nq,
              Nk, d, float(scale), int(window), _ptr(workspace), int(workspace_bytes), _stream(stream)),
           "fa_bwd_window")


def fa_fwd_varlen(q, k, v, o, lse, seqlens_q, seqlens_k, B, H, Nq, Nk, d, scale, causal, stream=None):
    fn = load().fa_fwd_varlen
    if fn.argtypes is None:
        vp, i = ctypes.c_void_p, ctypes.c_int
        fn.argtypes = [vp] * 7 + [i] * 5 + [ctypes.c_float, i, vp]
        fn.restype = i
    _raise(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(seqlens_q), _ptr(seqlens_k), B, H, Nq, Nk, d,
              float(scale), int(causal), _stream(stream)), "fa_fwd_varlen")


def fa_bwd_varlen(q, k, v, o, lse, dO, dq, dk, dv, seqlens_q, seqlens_k, B, H, Nq, Nk, d, scale, causal,
                  workspace, workspace_bytes, stream=None):
    fn = load().fa_bwd_varlen
    if fn.argtypes is None:
        vp, i = ctypes.c_void_p, ctypes.c_int
        fn.argtypes = [vp] * 11 + [i] * 5 + [ctypes.c_float, i, vp, ctypes.c_size_t, vp]
        fn.restype = i
    _raise(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv),
              _ptr(seqlens_q), _ptr(seqlens_k), B, H, Nq, Nk, d, float(scale), int(causal), _ptr(workspace),
              workspace_bytes, _stream(stream)), "fa_bwd_varlen")


def fa_fwd_fp8_workspace_bytes(B, H, Nk, d):
    fn = load().fa_fwd_fp8_workspace_bytes
    if fn.argtypes is None:
        fn.argtypes = [ctypes.c_int] * 4
        fn.restype = ctypes.c_size_t
    return fn(B, H, Nk, d)


def fa_fwd_fp8(q8, k8, v8, q_scale, k_scale, v_scale, o, lse, B, H, Nq, Nk, d, scale, causal, workspace,
               workspace_bytes, stream=None):
    fn = load().fa_fwd_fp8
    if fn.argtypes is None:
        vp, i = ctypes.c_void_p, ctypes.c_int
        fn.argtypes = [vp] * 8 + [i] * 5 + [ctypes.c_float, i, vp, ctypes.c_size_t, vp]
        fn.restype = i
    _raise(fn(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(q_scale), _ptr(k_scale), _ptr(v_scale), _ptr(o), _ptr(lse),
              B, H, Nq, Nk, d, float(scale), int(causal), _ptr(workspace), workspace_bytes, _stream(stream)),
           "fa_fwd_fp8")


def forward_fp8(q8, k8, v8, q_scale, k_scale, v_scale, scale=None, causal=False, stream=None, workspace=None):
    """O (bf16) and LSE for e4m3 q8 [B,H,Nq,128], k8/v8 [B,H,Nk,128] (uint8 CUDA tensors) with fp32
    scales: q_scale [B*H, ceil(Nq/128)], k_scale [B*H, ceil(Nk/128)], v_scale [B*H]."""
    B, H, Nq, d = q8.shape
    Nk = k8.shape[2]
    for t, n, shp in ((q8, "q8", (B, H, Nq, d)), (k8, "k8", (B, H, Nk, d)), (v8, "v8", (B, H, Nk, d))):
        if not (t.is_cuda and t.dtype == torch.uint8 and t.is_contiguous() and tuple(t.shape) == shp):
            raise ValueError("%s must be a contiguous uint8 CUDA tensor of shape %s" % (n, shp))
    for t, n, shp in ((q_scale, "q_scale", (B * H, -(-Nq // 128))), (k_scale, "k_scale", (B * H, -(-Nk // 128))),
                      (v_scale, "v_scale", (B * H,))):
        if not (t.is_cuda and t.dtype == torch.float32 and t.is_contiguous() and tuple(t.shape) == shp):
            raise ValueError("%s must be a contiguous float32 CUDA tensor of shape %s" % (n, shp))
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    nbytes = fa_fwd_fp8_workspace_bytes(B, H, Nk, d)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q8.device)
    o = torch.empty((B, H, Nq, d), dtype=torch.bfloat16, device=q8.device)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q8.device)
    fa_fwd_fp8(q8, k8, v8, q_scale, k_scale, v_scale, o, lse, B, H, Nq, Nk, d, scale, causal, workspace,
               workspace.numel() * workspace.element_size(), stream)
    return o, lse


def fa_selftest_wait_timeout(timeout_ns, stream=None):
    """Launch the watchdog self-test kernel (a wait that must run out)."""
    fn = load().fa_selftest_wait_timeout
    if fn.argtypes is None:
        fn.argtypes = [ctypes.c_uint64, ctypes.c_void_p]
        fn.restype = ctypes.c_int
    _raise(fn(int(timeout_ns), _stream(stream)), "fa_selftest_wait_timeout")


def fa_bwd_workspace_bytes(B, H, Nq, Nk, d):
    return int(load().fa_bwd_workspace_bytes(B, H, Nq, Nk, d))


def fa_decode_workspace_bytes(B, H, Nk, d, num_splits=0):
    return int(load().fa_decode_workspace_bytes(B, H, Nk, d, num_splits))


def fa_fwd(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, stream=None):
    _raise(load().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nk, d,
                         float(scale), int(bool(causal)), _stream(stream)), "fa_fwd")


def fa_work_schedule(n_items, chunk_items, grid, per_chunk):
    """The CTA that takes each work item in the persistent grids' static
    schedule (a list of n_items ints)."""
    owner = (ctypes.c_int * max(1, n_items))()
    _raise(load().fa_work_schedule(n_items, chunk_items, grid, int(bool(per_chunk)), owner), "fa_work_schedule")
    return list(owner)[:n_items]


def fa_fwd_tile_rows(B, H, Nq, Nk, d, causal):
    """Query rows per work tile fa_fwd takes for these sizes (256, or 128 for
    split-KV tiles)."""
    rows = load().fa_fwd_tile_rows(B, H, Nq, Nk, d, int(bool(causal)))
    if rows < 0:
        raise FAError(rows, "fa_fwd_tile_rows")
    return rows


def fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, Nq, Nk, d, scale, causal, workspace,
           workspace_bytes, stream=None):
    _raise(load().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq),
                         _ptr(dk), _ptr(dv), B, H, Nq, Nk, d, float(scale), int(bool(causal)),
                         _ptr(workspace), int(workspace_bytes), _stream(stream)), "fa_bwd")


def fa_bwd_fused_workspace_bytes(B, H, Nq, Nk, d):
    return load().fa_bwd_fused_workspace_bytes(B, H, Nq, Nk, d)


def fa_bwd_fused(q, k, v, o, lse, dO, dq, dk, dv, B, H, Nq, Nk, d, scale, causal, workspace,
                 workspace_bytes, stream=None):
    """fa_bwd in one pass over the key tiles (dQ by fp32 reduce-adds; d = 128)."""
    _raise(load().fa_bwd_fused(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk),
                               _ptr(dv), B, H, Nq, Nk, d, float(scale), int(causal), _ptr(workspace),
                               int(workspace_bytes), _stream(stream)), "fa_bwd_fused")


def fa_bwd_preprocess(o, dO, delta, B, H, Nq, d, stream=None):
    _raise(load().fa_bwd_preprocess(_ptr(o), _ptr(dO), _ptr(delta), B, H, Nq, d, _stream(stream)),
           "fa_bwd_preprocess")


def fa_bwd_dkdv(q, k, v, lse, delta, dO, dk, dv, B, H, Nq, Nk, d, scale, causal, stream=None):
    _raise(load().fa_bwd_dkdv(_ptr(q), _ptr(k), _ptr(v), _ptr(lse), _ptr(delta), _ptr(dO), _ptr(dk),
                              _ptr(dv), B, H, Nq, Nk, d, float(scale), int(bool(causal)),
                              _stream(stream)), "fa_bwd_dkdv")


def fa_bwd_dkdv_pair(q, k, v, lse, delta, dO, dk, dv, B, H, Nq, Nk, d, scale, causal, stream=None):
    """fa_bwd_dkdv on CTA pairs (cta_group::2 products; d = 128)."""
    _raise(load().fa_bwd_dkdv_pair(_ptr(q), _ptr(k), _ptr(v), _ptr(lse), _ptr(delta), _ptr(dO), _ptr(dk),
                                   _ptr(dv), B, H, Nq, Nk, d, float(scale), int(causal), _stream(stream)),
           "fa_bwd_dkdv_pair")


def fa_bwd_dq(q, k, v, lse, delta, dO, dq, B, H, Nq, Nk, d, scale, causal, stream=None):
    _raise(load().fa_bwd_dq(_ptr(q), _ptr(k), _ptr(v), _ptr(lse), _ptr(delta), _ptr(dO), _ptr(dq),
                            B, H, Nq, Nk, d, float(scale), int(bool(causal)), _stream(stream)),
           "fa_bwd_dq")


def fa_decode(q, kcache, vcache, o, lse, B, H, Nk, d, scale, num_splits, workspace,
              workspace_bytes, stream=None):
    _raise(load().fa_decode(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(o), _ptr(lse), B, H, Nk,
                            d, float(scale), int(num_splits), _ptr(workspace),
                            int(workspace_bytes), _stream(stream)), "fa_decode")


def fa_decode_noalloc(q, kcache, vcache, o, lse, B, H, Nk, d, scale, num_splits, stream=None):
    """fa_decode without a workspace: the partials go to the library's fixed
    scratch array (for callers that may not allocate; see include/fa.h)."""
    fn = load().fa_decode_noalloc
    if fn.argtypes is None:
        vp, i = ctypes.c_void_p, ctypes.c_int
        fn.argtypes = [vp] * 5 + [i, i, i, i, ctypes.c_float, i, vp]
        fn.restype = ctypes.c_int
    _raise(fn(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(o), _ptr(lse), B, H, Nk, d, float(scale),
              int(num_splits), _stream(stream)), "fa_decode_noalloc")


# ------------------------------------------------------------------ conveniences
def _check(t, name, shape):
    if not (t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()):
        raise ValueError("%s must be a contiguous bf16 CUDA tensor" % name)
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))


def _lens(t, B, name):
    if not (t.is_cuda and t.dtype == torch.int32 and t.is_contiguous() and t.shape == (B,)):
        raise ValueError("%s must be a contiguous int32 CUDA tensor of shape (%d,)" % (name, B))


def forward(q, k, v, scale=None, causal=False, stream=None, seqlens_q=None, seqlens_k=None):
    """O, LSE for q [B,H,Nq,d], k/v [B,H,Nk,d] (bf16 CUDA).  LSE is fp32 [B,H,Nq].

    With seqlens_q / seqlens_k (int32 [B] on the device, both or neither):
    per-sequence lengths within the padded tensors (fa_fwd_varlen)."""
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    _check(q, "q", (B, H, Nq, d))
    _check(k, "k", (B, H, Nk, d))
    _check(v, "v", (B, H, Nk, d))
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if seqlens_q is not None or seqlens_k is not None:
        _lens(seqlens_q, B, "seqlens_q")
        _lens(seqlens_k, B, "seqlens_k")
        fa_fwd_varlen(q, k, v, o, lse, seqlens_q, seqlens_k, B, H, Nq, Nk, d, scale, causal, stream)
    else:
        fa_fwd(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, stream)
    return o, lse


def backward(q, k, v, o, lse, dO, scale=None, causal=False, stream=None, workspace=None, seqlens_q=None,
             seqlens_k=None, fused=False):
    """dQ, dK, dV (bf16) for the forward output o / lse and upstream gradient dO.
    fused=True: fa_bwd_fused (one pass, dQ by fp32 reduce-adds; d = 128)."""
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    for t, n, s in ((q, "q", (B, H, Nq, d)), (k, "k", (B, H, Nk, d)), (v, "v", (B, H, Nk, d)),
                    (o, "o", (B, H, Nq, d)), (dO, "dO", (B, H, Nq, d))):
        _check(t, n, s)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    if fused and (seqlens_q is not None or seqlens_k is not None):
        raise ValueError("fused=True takes no sequence lengths")
    nbytes = (fa_bwd_fused_workspace_bytes if fused else fa_bwd_workspace_bytes)(B, H, Nq, Nk, d)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if seqlens_q is not None or seqlens_k is not None:
        _lens(seqlens_q, B, "seqlens_q")
        _lens(seqlens_k, B, "seqlens_k")
        fa_bwd_varlen(q, k, v, o, lse, dO, dq, dk, dv, seqlens_q, seqlens_k, B, H, Nq, Nk, d, scale, causal,
                      workspace, workspace.numel() * workspace.element_size(), stream)
    else:
        (fa_bwd_fused if fused else fa_bwd)(q, k, v, o, lse, dO, dq, dk, dv, B, H, Nq, Nk, d, scale, causal,
                                            workspace, workspace.numel() * workspace.element_size(), stream)
    return dq, dk, dv


def decode(q, kcache, vcache, scale=None, num_splits=0, stream=None, workspace=None,
           want_lse=True):
    """O [B,H,d] bf16 (and LSE [B,H] fp32) for one query per (b, h) against the caches."""
    B, H, d = q.shape
    Nk = kcache.shape[2]
    _check(q, "q", (B, H, d))
    _check(kcache, "kcache", (B, H, Nk, d))
    _check(vcache, "vcache", (B, H, Nk, d))
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    nbytes = fa_decode_workspace_bytes(B, H, Nk, d, num_splits)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    o = torch.empty_like(q)
    lse = torch.empty((B, H), dtype=torch.float32, device=q.device) if want_lse else None
    fa_decode(q, kcache, vcache, o, lse, B, H, Nk, d, scale, num_splits, workspace,
              workspace.numel() * workspace.element_size(), stream)
    return (o, lse) if want_lse else o
