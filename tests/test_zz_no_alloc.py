"""fa_decode_noalloc: split-KV decode whose partials live in the library's
fixed scratch array instead of a caller workspace, for callers that may not
allocate device memory (a plugin host that hands over only its input and
output buffers, a real-time loop that must not enter the allocator).

It is called through the C ABI and checked against fa_decode (the entry point
with a workspace) on two calls in a row, with the parity tolerances of the
other decode tests.  This file is collected last on purpose.
"""
import ctypes
import math

import pytest
import torch

import exact_tiled_attention_21_gb300 as fa
from exact_tiled_attention_21_gb300 import synthetic as syn
from tests.parity import check_out, f64

pytestmark = pytest.mark.gpu

LIMIT = 16 << 20  # FA_DECODE_NOALLOC_SCRATCH_BYTES in include/fa.h


def _case(seed, B, H, Nk, d):
    dev = torch.device("cuda", 0)
    return (syn.bhd(seed, syn.TAG_Q, B, H, d).to(dev), syn.bhnd(seed, syn.TAG_K, B, H, Nk, d).to(dev),
            syn.bhnd(seed, syn.TAG_V, B, H, Nk, d).to(dev))


def _with_workspace(q, kc, vc, scale, splits):
    B, H, d = q.shape
    Nk = kc.shape[2]
    o = torch.empty_like(q)
    lse = torch.empty(B, H, device=q.device, dtype=torch.float32)
    ws = torch.empty(fa.fa_decode_workspace_bytes(B, H, Nk, d, splits), dtype=torch.uint8, device=q.device)
    fa.fa_decode(q, kc, vc, o, lse, B, H, Nk, d, scale, splits, ws, ws.numel())
    return o, lse


def _no_alloc(q, kc, vc, scale, splits):
    B, H, d = q.shape
    Nk = kc.shape[2]
    o = torch.empty_like(q)
    lse = torch.empty(B, H, device=q.device, dtype=torch.float32)
    fa.fa_decode_noalloc(q, kc, vc, o, lse, B, H, Nk, d, scale, splits)
    return o, lse


def test_no_alloc_decode_matches_workspace_decode_twice(cuda_lib):
    # two calls in a row with different shapes: the second sees the first's
    # partials still in the shared array and must not depend on them
    for seed, (B, H, Nk, d, splits) in ((41, (32, 32, 4096, 128, 16)), (42, (3, 5, 1000, 64, 7))):
        q, kc, vc = _case(seed, B, H, Nk, d)
        scale = 1.0 / math.sqrt(d)
        o_ref, lse_ref = _with_workspace(q, kc, vc, scale, splits)
        o, lse = _no_alloc(q, kc, vc, scale, splits)
        torch.cuda.synchronize()
        check_out(f64(o.cpu()), f64(lse.cpu()), f64(o_ref.cpu()), f64(lse_ref.cpu()),
                  "no-alloc vs workspace B%d H%d Nk%d d%d S%d" % (B, H, Nk, d, splits))


def test_no_alloc_decode_rejects_problems_beyond_the_scratch(cuda_lib):
    B, H, Nk, d, splits = 64, 64, 4096, 128, 16  # partials need 32 MiB + 256 KiB
    assert fa.fa_decode_workspace_bytes(B, H, Nk, d, splits) > LIMIT
    vp = ctypes.c_void_p
    lib = fa.load()
    with pytest.raises(fa.FAError) as err:
        fa.fa_decode_noalloc(None, None, None, None, None, B, H, Nk, d, 0.1, splits)
    assert err.value.status == fa.FA_ERR_INVALID_ARG  # null pointers are checked first
    # argtypes were set by the binding's first call above; the pointers are
    # never dereferenced because the size check comes before any launch
    st = lib.fa_decode_noalloc(vp(256), vp(256), vp(256), vp(256), None, B, H, Nk, d, 0.1, splits, None)
    assert st == fa.FA_ERR_WORKSPACE
