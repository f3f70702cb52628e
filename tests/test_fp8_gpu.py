"""FP8 block-scaled forward (fa_fwd_fp8) against the fp64 oracle on the
dequantised inputs (oracle.naive.forward_fp8), with the rounding bound of
tests.parity.check_out_fp8."""
import math

import numpy as np
import pytest
import torch

from exact_tiled_attention_21_gb300 import synthetic as syn
from oracle import naive
from tests.parity import check_out_fp8

pytestmark = pytest.mark.gpu


def _inputs(seed, B, H, Nq, Nk, heads=None, k_ramp=None):
    heads = range(H) if heads is None else heads

    def gen(tag, n):
        x = torch.zeros(B, H, n, 128)
        for b in range(B):
            for h in heads:
                x[b, h] = syn.head_f32(seed, tag, b, h, n, 128)
        return x
    q8, sq = syn.to_e4m3(gen(syn.TAG_Q, Nq), rows=128)
    k = gen(syn.TAG_K, Nk)
    if k_ramp is not None:  # key row t scaled by k_ramp[t] before quantisation
        k = k * k_ramp[None, None, :, None]
    k8, sk = syn.to_e4m3(k, rows=128)
    v8, sv = syn.to_e4m3(gen(syn.TAG_V, Nk))
    return q8, k8, v8, sq, sk, sv


def _run(fa, q8, k8, v8, sq, sk, sv, causal):
    dev = torch.device("cuda", 0)
    o, lse = fa.forward_fp8(*(t.to(dev) for t in (q8, k8, v8, sq, sk, sv)), causal=causal)
    torch.cuda.synchronize()
    st, detail = fa.fa_get_last_device_error()
    assert st == 0, detail
    return o.cpu(), lse.cpu()


def _oracle(q8, k8, v8, sq, sk, sv, causal, rows=None, Nq=None, heads=None):
    qn, kn, vn = q8.numpy(), k8.numpy(), v8.numpy()
    v = naive.dequant_e4m3(vn, sv.numpy())
    q = naive.dequant_e4m3(qn, sq.numpy(), rows=128)
    k = naive.dequant_e4m3(kn, sk.numpy(), rows=128)
    if rows is not None:
        q = q[:, :, rows]
    o, lse, p = naive.forward(q, k, v, 1 / math.sqrt(128), causal, rows=rows, Nq=Nq, return_p=True)
    o2, lse2 = naive.forward_fp8(qn if rows is None else qn[:, :, rows], kn, vn, sq.numpy(), sk.numpy(),
                                 sv.numpy(), 1 / math.sqrt(128), causal, rows=rows, Nq=Nq)
    np.testing.assert_array_equal(o, o2)  # the oracle's own two routes agree
    return o, lse, p, v


# (B, H, Nq, Nk, causal)
CASES = [
    (1, 2, 1000, 1000, False),
    (1, 2, 1000, 1000, True),
    (1, 2, 700, 1300, True),
    (1, 2, 1300, 700, True),     # the first 600 rows see no key
    (1, 2, 2048, 2048, False),
    (2, 3, 513, 513, True),
    (1, 1, 1, 37, False),
]


@pytest.mark.parametrize("B,H,Nq,Nk,causal", CASES)
def test_fp8_forward_parity(cuda_lib, B, H, Nq, Nk, causal):
    q8, k8, v8, sq, sk, sv = _inputs(2100 + Nq + Nk, B, H, Nq, Nk)
    o, lse = _run(cuda_lib, q8, k8, v8, sq, sk, sv, causal)
    o_ref, lse_ref, p_ref, v = _oracle(q8, k8, v8, sq, sk, sv, causal)
    check_out_fp8(o.double().numpy(), lse.double().numpy(), o_ref, lse_ref, p_ref, v,
                  "fp8 Nq%d Nk%d causal%d" % (Nq, Nk, causal))


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_growing_scores(cuda_lib, causal):
    """Key rows scaled by a ramp (0.5 at the first key to 12.5 at the last, the
    per-block scales following it): the row max grows by more than 2^8 in the
    log2 domain every block or two, so blocks whose exponentials ran against
    the running max are redone after the accumulator is rescaled."""
    Nq = Nk = 1024
    ramp = 0.5 + 12.0 * torch.arange(Nk, dtype=torch.float32) / Nk
    q8, k8, v8, sq, sk, sv = _inputs(2500, 1, 2, Nq, Nk, k_ramp=ramp)
    o, lse = _run(cuda_lib, q8, k8, v8, sq, sk, sv, causal)
    o_ref, lse_ref, p_ref, v = _oracle(q8, k8, v8, sq, sk, sv, causal)
    check_out_fp8(o.double().numpy(), lse.double().numpy(), o_ref, lse_ref, p_ref, v,
                  "fp8 growing scores causal%d" % causal)


def test_fp8_forward_full_size_sampled(cuda_lib):
    """B=1, H=32, N=8192, causal (the bench workload): 8 heads x 256 seeded rows
    (always including rows 0 and N - 1)."""
    N, H = 8192, 32
    heads = syn.sample_heads(31, H, 8)
    q8, k8, v8, sq, sk, sv = _inputs(4242, 1, H, N, N, heads=heads)
    o, lse = _run(cuda_lib, q8, k8, v8, sq, sk, sv, True)
    rows = syn.sample_rows(31, N, 256)
    for h in heads:
        sl = slice(h, h + 1)
        o_ref, lse_ref, p_ref, v = _oracle(q8[:, sl], k8[:, sl], v8[:, sl], sq[sl], sk[sl], sv[sl], True,
                                           rows=rows, Nq=N)
        check_out_fp8(o[:, sl][:, :, rows].double().numpy(), lse[:, sl][:, :, rows].double().numpy(), o_ref,
                      lse_ref, p_ref, v, "fp8 full size head %d" % h)


def test_fp8_rejects_d64(cuda_lib):
    fa = cuda_lib
    dev = torch.device("cuda", 0)
    x = torch.zeros(1, 1, 8, 64, dtype=torch.uint8, device=dev)
    with pytest.raises(fa.FAError):
        fa.fa_fwd_fp8(x, x, x, torch.ones(1, 1, device=dev), torch.ones(1, 1, device=dev),
                      torch.ones(1, device=dev), torch.empty(1, 1, 8, 64, dtype=torch.bfloat16, device=dev),
                      torch.empty(1, 1, 8, device=dev), 1, 1, 8, 8, 64, 0.125, 0,
                      torch.empty(4096, dtype=torch.uint8, device=dev), 4096)


def test_fp8_output_16_byte_aligned(cuda_lib):
    """O written 16 bytes past a 32-byte boundary takes the 16-byte store path:
    the same bits as an aligned O."""
    fa = cuda_lib
    dev = torch.device("cuda", 0)
    B, H, N = 1, 2, 700
    q8, k8, v8, sq, sk, sv = (t.to(dev) for t in _inputs(2333, B, H, N, N))
    o_ref, lse_ref = fa.forward_fp8(q8, k8, v8, sq, sk, sv, causal=True)
    buf = torch.empty(B * H * N * 128 + 16, dtype=torch.bfloat16, device=dev)
    start = ((16 - buf.data_ptr() % 32) % 32) // 2
    o = buf[start:start + B * H * N * 128].view(B, H, N, 128)
    assert o.data_ptr() % 32 == 16
    lse = torch.empty(B, H, N, device=dev)
    ws = torch.empty(fa.fa_fwd_fp8_workspace_bytes(B, H, N, 128), dtype=torch.uint8, device=dev)
    fa.fa_fwd_fp8(q8, k8, v8, sq, sk, sv, o, lse, B, H, N, N, 128, 1 / math.sqrt(128), True, ws, ws.numel())
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_error()[0] == 0
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
