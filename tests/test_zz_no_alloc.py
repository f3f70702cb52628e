"""fa_decode_noalloc: split-KV decode whose partials live in the library's
fixed scratch array instead of a caller workspace, for callers that may not
allocate device memory (a plugin host that hands over only its input and
output buffers, a real-time loop that must not enter the allocator).

It is called through the C ABI.  It runs the same kernels with the same split
count as fa_decode (the entry point with a workspace) and writes its partials
in the same layout, so its outputs must equal fa_decode's bit for bit; each
case is also checked against the fp64 oracle.  Every call shares the array,
so the tests also run a call whose partials are all NaN right before a clean
call of the same shape: the clean call must not see them.  This file is
collected last on purpose.
"""
import math

import pytest
import torch

import exact_tiled_attention_21_gb300 as fa
from exact_tiled_attention_21_gb300 import synthetic as syn
from oracle import naive
from tests.parity import check_out, f64

pytestmark = pytest.mark.gpu

LIMIT = 16 << 20  # FA_DECODE_NOALLOC_SCRATCH_BYTES in include/fa.h


def _case(seed, B, H, Nk, d):
    return (syn.bhd(seed, syn.TAG_Q, B, H, d), syn.bhnd(seed, syn.TAG_K, B, H, Nk, d),
            syn.bhnd(seed, syn.TAG_V, B, H, Nk, d))


def _dev(*ts):
    dev = torch.device("cuda", 0)
    return tuple(t.to(dev) for t in ts)


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


def _check(q, kc, vc, scale, splits, what):
    """fa_decode_noalloc equals fa_decode bit for bit and the oracle within tolerance."""
    qd, kd, vd = _dev(q, kc, vc)
    o, lse = _no_alloc(qd, kd, vd, scale, splits)
    o_ref, lse_ref = _with_workspace(qd, kd, vd, scale, splits)
    torch.cuda.synchronize()
    assert torch.isfinite(o).all(), "%s: non-finite output" % what
    assert torch.equal(o, o_ref), "%s: O differs from fa_decode" % what
    assert torch.equal(lse, lse_ref), "%s: LSE differs from fa_decode" % what
    oo, ll = naive.decode(f64(q), f64(kc), f64(vc), scale)
    check_out(f64(o.cpu()), f64(lse.cpu()), oo, ll, what)


def test_no_alloc_decode_matches_workspace_decode_twice(cuda_lib):
    # two calls in a row: the B=32, H=32, Nk=4096 workload on the tensor-core
    # kernel, then a short d=64 cache on the 16-byte-load kernel
    for seed, (B, H, Nk, d, splits) in ((41, (32, 32, 4096, 128, 16)), (42, (3, 5, 100, 64, 7))):
        q, kc, vc = _case(seed, B, H, Nk, d)
        _check(q, kc, vc, 1.0 / math.sqrt(d), splits, "B%d H%d Nk%d d%d S%d" % (B, H, Nk, d, splits))


@pytest.mark.parametrize("B,H,Nk,d,splits", [(4, 8, 1024, 128, 8), (4, 8, 1000, 64, 8), (4, 8, 100, 128, 8)])
def test_no_alloc_decode_ignores_stale_partials(cuda_lib, B, H, Nk, d, splits):
    # same shape twice: the first call's V is all NaN, so every partial slot it
    # writes in the shared array holds NaN; the second, clean call must not read
    # any of them (the first shape runs on the tensor-core kernel, the other two
    # on the 16-byte-load kernel)
    q, kc, vc = _case(43 + d, B, H, Nk, d)
    scale = 1.0 / math.sqrt(d)
    qd, kd = _dev(q, kc)
    vnan = torch.full((B, H, Nk, d), float("nan"), dtype=torch.bfloat16, device=qd.device)
    o_nan, _ = _no_alloc(qd, kd, vnan, scale, splits)
    torch.cuda.synchronize()
    assert torch.isnan(o_nan).all()
    _check(q, kc, vc, scale, splits, "after a NaN call B%d H%d Nk%d d%d S%d" % (B, H, Nk, d, splits))


def test_no_alloc_decode_rejects_problems_beyond_the_scratch(cuda_lib):
    with pytest.raises(fa.FAError) as err:
        fa.fa_decode_noalloc(None, None, None, None, None, 1, 1, 128, 128, 0.1, 1)
    assert err.value.status == fa.FA_ERR_INVALID_ARG  # null pointers are checked first
    # real buffers: 16 x 16 heads, 256 keys, 256 splits need 32 MiB + 256 KiB of partials
    B, H, Nk, d, splits = 16, 16, 256, 128, 256
    assert fa.fa_decode_workspace_bytes(B, H, Nk, d, splits) > LIMIT
    q, kc, vc = _dev(*_case(44, B, H, Nk, d))
    with pytest.raises(fa.FAError) as err:
        _no_alloc(q, kc, vc, 1.0 / math.sqrt(d), splits)
    assert err.value.status == fa.FA_ERR_WORKSPACE
    # the same problem with fewer splits fits and still runs
    _check(*_case(44, B, H, Nk, d), 1.0 / math.sqrt(d), 16, "B16 H16 Nk256 S16 after the rejection")
