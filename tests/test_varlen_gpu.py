"""Per-sequence lengths in a padded batch (fa_fwd_varlen / fa_bwd_varlen)
against the fp64 oracle (oracle.naive.forward_varlen / backward_varlen)."""
import math

import numpy as np
import pytest
import torch

import exact_tiled_attention_21_gb300 as fa_mod
from exact_tiled_attention_21_gb300 import synthetic as syn
from oracle import naive
from tests.parity import check_grad, check_out, f64

pytestmark = pytest.mark.gpu

# (H, Nq, Nk, d, causal, lens_q, lens_k): B = len(lens_q)
CASES = [
    (2, 700, 700, 128, True, [700, 513, 129, 1], [700, 513, 129, 1]),
    (2, 700, 700, 128, False, [700, 300, 0, 129], [64, 700, 5, 640]),
    (2, 300, 900, 64, True, [300, 17, 256, 1], [900, 1, 500, 256]),   # Nk > Nq: queries at the end
    (2, 900, 300, 128, True, [900, 300, 40, 600], [300, 300, 200, 1]),  # rows that see no key
    (3, 256, 256, 64, False, [256, 255], [128, 129]),
    # many heads; key tiles of empty sequences (no query tile, dK = dV = 0) among
    # the others
    (40, 384, 384, 64, True, [384, 100, 0, 257], [384, 128, 0, 300]),
]


def _padded(seed, B, H, Nq, Nk, d, lq, lk):
    """Inputs whose padding positions hold large finite values (they must not
    matter), and the same inputs with zero padding for the oracle."""
    q, k, v, dO = (syn.bhnd(seed, syn.TAG_Q, B, H, Nq, d), syn.bhnd(seed, syn.TAG_K, B, H, Nk, d),
                   syn.bhnd(seed, syn.TAG_V, B, H, Nk, d), syn.bhnd(seed, syn.TAG_DO, B, H, Nq, d))
    clean = [t.clone() for t in (q, k, v, dO)]
    for b in range(B):
        for t, n, fill in ((q, lq[b], 40.0), (k, lk[b], -30.0), (v, lk[b], 50.0), (dO, lq[b], 20.0)):
            t[b, :, n:] = fill
        for t, n in ((clean[0], lq[b]), (clean[1], lk[b]), (clean[2], lk[b]), (clean[3], lq[b])):
            t[b, :, n:] = 0
    return (q, k, v, dO), clean


def _run(fa, q, k, v, dO, lq, lk, causal, scale):
    dev = torch.device("cuda", 0)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    qd, kd, vd, dOd = (t.to(dev) for t in (q, k, v, dO))
    lqd = torch.tensor(lq, dtype=torch.int32, device=dev)
    lkd = torch.tensor(lk, dtype=torch.int32, device=dev)
    o, lse = fa.forward(qd, kd, vd, scale, causal, seqlens_q=lqd, seqlens_k=lkd)
    dq, dk, dv = fa.backward(qd, kd, vd, o, lse, dOd, scale, causal, seqlens_q=lqd, seqlens_k=lkd)
    torch.cuda.synchronize()
    st, detail = fa.fa_get_last_device_error()
    assert st == 0, detail
    return [t.cpu() for t in (o, lse, dq, dk, dv)]


@pytest.mark.parametrize("H,Nq,Nk,d,causal,lq,lk", CASES)
def test_varlen_forward_backward_parity(cuda_lib, H, Nq, Nk, d, causal, lq, lk):
    B = len(lq)
    scale = 1 / math.sqrt(d)
    (q, k, v, dO), clean = _padded(1700 + Nq + Nk + d, B, H, Nq, Nk, d, lq, lk)
    o, lse, dq, dk, dv = _run(cuda_lib, q, k, v, dO, lq, lk, causal, scale)
    tag = "Nq%d Nk%d d%d causal%d" % (Nq, Nk, d, causal)
    cq, ck, cv, cdo = (f64(t) for t in clean)
    o_ref, lse_ref = naive.forward_varlen(cq, ck, cv, lq, lk, scale, causal)
    check_out(f64(o), f64(lse), o_ref, lse_ref, "fwd " + tag)
    rq, rk, rv = naive.backward_varlen(cq, ck, cv, cdo, lq, lk, scale, causal)
    dp_max = np.abs(cdo @ np.swapaxes(cv, -1, -2)).max()
    cancel = scale * dp_max * max(np.abs(ck).max(), np.abs(cq).max())
    check_grad(f64(dq), rq, "dQ " + tag, cancel_scale=cancel)
    check_grad(f64(dk), rk, "dK " + tag, cancel_scale=cancel)
    check_grad(f64(dv), rv, "dV " + tag)
    for b in range(B):  # padding rows are exact zeros (and -inf LSE)
        assert (o[b, :, lq[b]:] == 0).all() and torch.isneginf(lse[b, :, lq[b]:]).all()
        assert (dq[b, :, lq[b]:] == 0).all()
        assert (dk[b, :, lk[b]:] == 0).all() and (dv[b, :, lk[b]:] == 0).all()


def test_varlen_full_lengths_match_dense(cuda_lib):
    """Lengths equal to the padded sizes give bit-identical results to fa_fwd /
    fa_bwd (the same tiles, in the same order).  Enough heads that fa_fwd takes
    256-row tiles, as the per-sequence-length forward always does."""
    fa = cuda_lib
    B, H, N, d = 2, 80, 640, 128
    assert fa.fa_fwd_tile_rows(B, H, N, N, d, 0) == 256 and fa.fa_fwd_tile_rows(B, H, N, N, d, 1) == 256
    q, k, v, dO = (syn.bhnd(77, t, B, H, N, d).cuda() for t in (syn.TAG_Q, syn.TAG_K, syn.TAG_V, syn.TAG_DO))
    lens = torch.full((B,), N, dtype=torch.int32, device=q.device)
    for causal in (False, True):
        o1, l1 = fa.forward(q, k, v, causal=causal)
        o2, l2 = fa.forward(q, k, v, causal=causal, seqlens_q=lens, seqlens_k=lens)
        g1 = fa.backward(q, k, v, o1, l1, dO, causal=causal)
        g2 = fa.backward(q, k, v, o2, l2, dO, causal=causal, seqlens_q=lens, seqlens_k=lens)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
        for a, b in zip(g1, g2):
            assert torch.equal(a, b)


def test_varlen_length_out_of_range_is_recorded(cuda_lib):
    """A length above the padded size is clamped (never read past the tensor)
    and recorded as FA_ERR_INVALID_ARG in the device error word."""
    fa = cuda_lib
    dev = torch.device("cuda", 0)
    B, H, N, d = 2, 1, 256, 64
    q = syn.bhnd(3, syn.TAG_Q, B, H, N, d).to(dev)
    lq = torch.tensor([N + 100, 10], dtype=torch.int32, device=dev)
    lk = torch.tensor([N, 10], dtype=torch.int32, device=dev)
    o, lse = fa.forward(q, q, q, seqlens_q=lq, seqlens_k=lk)
    st, detail = fa.fa_get_last_device_error()
    assert st == fa_mod.FA_ERR_INVALID_ARG, detail
    o2, lse2 = fa.forward(q, q, q, seqlens_q=torch.tensor([N, 10], dtype=torch.int32, device=dev), seqlens_k=lk)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    assert fa.fa_get_last_device_error()[0] == 0


def test_varlen_rejects_null_lengths(cuda_lib):
    fa = cuda_lib
    dev = torch.device("cuda", 0)
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(1, 1, 8, device=dev)
    lens = torch.tensor([8], dtype=torch.int32, device=dev)
    with pytest.raises(fa.FAError):
        fa.fa_fwd_varlen(q, q, q, torch.empty_like(q), lse, lens, None, 1, 1, 8, 8, 64, 0.125, 0)
