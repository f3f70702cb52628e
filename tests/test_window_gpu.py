"""Causal sliding-window attention (fa_fwd_window / fa_bwd_window) against the
fp64 oracle with the same window."""
import math

import numpy as np
import pytest
import torch

from exact_tiled_attention_21_gb300 import synthetic as syn
from oracle import naive
from tests.parity import check_grad, check_out, f64

pytestmark = pytest.mark.gpu

# (B, H, Nq, Nk, d, window)
CASES = [
    (1, 2, 1000, 1000, 128, 256),
    (1, 2, 700, 1200, 64, 100),     # queries see a window ending at i + 500
    (1, 2, 1200, 700, 128, 1),      # one key per row; the first 500 rows see none
    (1, 2, 2048, 2048, 128, 512),
    (1, 2, 300, 300, 128, 4096),    # wider than the sequence: plain causal
    (2, 3, 513, 513, 64, 130),
    (1, 2, 1000, 1000, 128, 128),   # windows of at most 128 keys take split-KV tiles
    (2, 2, 777, 1300, 128, 37),
    (1, 3, 1100, 900, 64, 128),
    (1, 2, 1024, 1024, 128, 129),   # the widest window that takes split-KV tiles
]


def _inputs(seed, B, H, Nq, Nk, d):
    return (syn.bhnd(seed, syn.TAG_Q, B, H, Nq, d), syn.bhnd(seed, syn.TAG_K, B, H, Nk, d),
            syn.bhnd(seed, syn.TAG_V, B, H, Nk, d), syn.bhnd(seed, syn.TAG_DO, B, H, Nq, d))


@pytest.mark.parametrize("B,H,Nq,Nk,d,w", CASES)
def test_window_forward_backward_parity(cuda_lib, B, H, Nq, Nk, d, w):
    fa = cuda_lib
    q, k, v, dO = _inputs(1300 + Nq + Nk + w, B, H, Nq, Nk, d)
    scale = 1 / math.sqrt(d)
    dev = torch.device("cuda", 0)
    qd, kd, vd, dOd = (t.to(dev) for t in (q, k, v, dO))
    o = torch.empty_like(qd)
    lse = torch.empty(B, H, Nq, device=dev)
    fa.fa_fwd_window(qd, kd, vd, o, lse, B, H, Nq, Nk, d, scale, w)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, Nq, Nk, d), dtype=torch.uint8, device=dev)
    fa.fa_bwd_window(qd, kd, vd, o, lse, dOd, dq, dk, dv, B, H, Nq, Nk, d, scale, w, ws, ws.numel())
    torch.cuda.synchronize()
    st, detail = fa.fa_get_last_device_error()
    assert st == 0, detail
    tag = "Nq%d Nk%d d%d w%d" % (Nq, Nk, d, w)
    o_ref, lse_ref = naive.forward(f64(q), f64(k), f64(v), scale, True, window=w)
    check_out(f64(o.cpu()), f64(lse.cpu()), o_ref, lse_ref, "fwd " + tag)
    rq, rk, rv = naive.backward(f64(q), f64(k), f64(v), f64(dO), scale, True, window=w)
    dp_max = np.abs(f64(dO) @ np.swapaxes(f64(v), -1, -2)).max()
    cancel = scale * dp_max * max(np.abs(f64(k)).max(), np.abs(f64(q)).max())
    check_grad(f64(dq.cpu()), rq, "dQ " + tag, cancel_scale=cancel)
    check_grad(f64(dk.cpu()), rk, "dK " + tag, cancel_scale=cancel)
    check_grad(f64(dv.cpu()), rv, "dV " + tag)


def test_window_rejects_nonpositive_window(cuda_lib):
    fa = cuda_lib
    dev = torch.device("cuda", 0)
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(1, 1, 8, device=dev)
    with pytest.raises(fa.FAError):
        fa.fa_fwd_window(q, q, q, torch.empty_like(q), lse, 1, 1, 8, 8, 64, 0.125, 0)
