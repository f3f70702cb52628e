"""Backward parity: dQ, dK, dV from the CUDA path (fed with the CUDA forward's
O and LSE) against the fp64 oracle's exact gradients of the same inputs."""
import math

import numpy as np

import pytest
import torch

from exact_tiled_attention_21_gb300 import synthetic as syn
from oracle import naive
from tests.parity import check_grad, check_out, f64

pytestmark = pytest.mark.gpu


def _inputs(seed, B, H, Nq, Nk, d):
    return (syn.bhnd(seed, syn.TAG_Q, B, H, Nq, d), syn.bhnd(seed, syn.TAG_K, B, H, Nk, d),
            syn.bhnd(seed, syn.TAG_V, B, H, Nk, d), syn.bhnd(seed, syn.TAG_DO, B, H, Nq, d))


def _run(fa, q, k, v, dO, scale, causal, fused=False):
    dev = torch.device("cuda", 0)
    qd, kd, vd, dOd = (t.to(dev) for t in (q, k, v, dO))
    o, lse = fa.forward(qd, kd, vd, scale=scale, causal=causal)
    dq, dk, dv = fa.backward(qd, kd, vd, o, lse, dOd, scale=scale, causal=causal, fused=fused)
    torch.cuda.synchronize()
    st, detail = fa.fa_get_last_device_error()
    assert st == 0, detail
    return dq.cpu(), dk.cpu(), dv.cpu()


CASES = [
    (1, 2, 128, 128, 64, False),
    (1, 2, 128, 128, 64, True),
    (1, 2, 300, 300, 128, True),
    (1, 2, 1000, 1000, 128, False),
    (1, 2, 1000, 1000, 64, True),
    (2, 2, 513, 257, 128, False),
    (1, 2, 257, 513, 128, True),
    (1, 2, 200, 700, 128, True),     # every query sees a prefix of >= 500 keys
    (1, 2, 700, 200, 128, True),     # the first 500 queries see no key: zero dQ rows
    (1, 1, 1, 1, 64, False),
    (1, 2, 1, 300, 128, False),
    (1, 2, 300, 1, 64, True),
    (2, 3, 77, 1031, 64, True),
    (1, 2, 128, 128, 128, True),
    (1, 2, 128, 128, 128, False),
    (1, 2, 300, 1, 128, False),
    (3, 2, 129, 129, 128, True),
    (1, 3, 640, 384, 128, True),
]


FUSED_CASES = [c + (True,) for c in CASES if c[4] == 128]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,fused", [c + (False,) for c in CASES] + FUSED_CASES)
def test_backward_parity(cuda_lib, B, H, Nq, Nk, d, causal, fused):
    """fa_bwd (two passes) and fa_bwd_fused (one pass, dQ by fp32 reduce-adds)."""
    seed = 500 + Nq * 3 + Nk + d + causal
    q, k, v, dO = _inputs(seed, B, H, Nq, Nk, d)
    scale = 1.0 / math.sqrt(d)
    dq, dk, dv = _run(cuda_lib, q, k, v, dO, scale, causal, fused)
    rq, rk, rv = naive.backward(f64(q), f64(k), f64(v), f64(dO), scale, causal)
    tag = "B%d H%d Nq%d Nk%d d%d c%d%s" % (B, H, Nq, Nk, d, causal, " fused" if fused else "")
    dp_max = np.abs(f64(dO) @ np.swapaxes(f64(v), -1, -2)).max()
    cancel = scale * dp_max * max(np.abs(f64(k)).max(), np.abs(f64(q)).max())
    check_grad(f64(dq), rq, "dQ " + tag, cancel_scale=cancel)
    check_grad(f64(dk), rk, "dK " + tag, cancel_scale=cancel)
    check_grad(f64(dv), rv, "dV " + tag)


# Many heads at small N, every head checked: grids of several waves of CTAs
# (B*H = the SM count, times the key or query tiles per head).
MANY_HEAD_CASES = [
    (384, 384, 64, True),
    (200, 256, 128, False),   # ragged query tail
]


@pytest.mark.parametrize("Nq,Nk,d,causal", MANY_HEAD_CASES)
def test_backward_parity_many_heads(cuda_lib, Nq, Nk, d, causal):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B, H = (2, sms // 2) if sms % 2 == 0 else (1, sms)
    seed = 900 + Nq * 3 + Nk + d + causal
    q, k, v, dO = _inputs(seed, B, H, Nq, Nk, d)
    scale = 1.0 / math.sqrt(d)
    dq, dk, dv = _run(cuda_lib, q, k, v, dO, scale, causal)
    rq, rk, rv = naive.backward(f64(q), f64(k), f64(v), f64(dO), scale, causal)
    tag = "B%d H%d Nq%d Nk%d d%d c%d" % (B, H, Nq, Nk, d, causal)
    dp_max = np.abs(f64(dO) @ np.swapaxes(f64(v), -1, -2)).max()
    cancel = scale * dp_max * max(np.abs(f64(k)).max(), np.abs(f64(q)).max())
    check_grad(f64(dq), rq, "dQ " + tag, cancel_scale=cancel)
    check_grad(f64(dk), rk, "dK " + tag, cancel_scale=cancel)
    check_grad(f64(dv), rv, "dV " + tag)


def test_backward_schedule_with_chunks_smaller_than_the_grid(cuda_lib):
    """B=1, H=32, Nq=16384, Nk=512, causal: the dK/dV pass's L2 chunks (8 heads
    of 4 key tiles) are smaller than its grid, so the persistent CTAs take the
    items in rounds over the whole list instead of per chunk; the dQ pass keeps
    per-chunk rounds.  Heads 0 and 31 against the oracle (queries before
    16384 - 512 see no key: zero dQ rows)."""
    B, H, Nq, Nk, d = 1, 32, 16384, 512, 128
    q, k, v, dO = _inputs(77, B, H, Nq, Nk, d)
    scale = 1.0 / math.sqrt(d)
    dq, dk, dv = _run(cuda_lib, q, k, v, dO, scale, True)
    for h in (0, H - 1):
        sl = slice(h, h + 1)
        rq, rk, rv = naive.backward(f64(q[:, sl]), f64(k[:, sl]), f64(v[:, sl]), f64(dO[:, sl]), scale, True)
        tag = "Nq%d Nk%d head %d" % (Nq, Nk, h)
        dp_max = np.abs(f64(dO[:, sl]) @ np.swapaxes(f64(v[:, sl]), -1, -2)).max()
        cancel = scale * dp_max * max(np.abs(f64(k[:, sl])).max(), np.abs(f64(q[:, sl])).max())
        check_grad(f64(dq[:, sl]), rq, "dQ " + tag, cancel_scale=cancel)
        check_grad(f64(dk[:, sl]), rk, "dK " + tag, cancel_scale=cancel)
        check_grad(f64(dv[:, sl]), rv, "dV " + tag)


@pytest.mark.parametrize("B,H,N", [(1, 1, 128), (1, 2, 700), (1, 32, 2048)])
def test_backward_matches_step_entry_points(cuda_lib, B, H, N):
    """fa_bwd launches the dQ pass to overlap the end of the dK/dV pass: the
    same kernels as the three step entry points, so the same bits; and work
    queued on the stream right after fa_bwd sees finished dK and dV (the dQ
    grid completes only after the dK/dV grid)."""
    fa = cuda_lib
    dev = torch.device("cuda", 0)
    d = 128
    q, k, v, dO = (t.to(dev) for t in _inputs(31 + N, B, H, N, N, d))
    o, lse = fa.forward(q, k, v, causal=True)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, N, d), dtype=torch.uint8, device=dev)
    dq1, dk1, dv1 = torch.empty_like(q), torch.full_like(k, float("nan")), torch.full_like(v, float("nan"))
    fa.fa_bwd(q, k, v, o, lse, dO, dq1, dk1, dv1, B, H, N, N, d, d ** -0.5, True, ws, ws.numel())
    dk_seen, dv_seen = dk1.clone(), dv1.clone()  # queued right behind fa_bwd, no synchronisation between
    delta = torch.empty(B, H, N, device=dev)
    dq2, dk2, dv2 = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fa.fa_bwd_preprocess(o, dO, delta, B, H, N, d)
    fa.fa_bwd_dkdv(q, k, v, lse, delta, dO, dk2, dv2, B, H, N, N, d, d ** -0.5, True)
    fa.fa_bwd_dq(q, k, v, lse, delta, dO, dq2, B, H, N, N, d, d ** -0.5, True)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_error()[0] == 0
    assert torch.equal(dq1, dq2) and torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    assert torch.equal(dk_seen, dk2) and torch.equal(dv_seen, dv2)


def test_backward_back_to_back_on_one_workspace(cuda_lib):
    """Three fa_bwd calls queued back to back on one workspace (filled with 0xFF
    bytes first): each call's preprocess overwrites D only after the dQ pass of
    the call before it, which still reads D, is done, so every call gives the
    bits of the three step entry points.  B=2, H=32, N=1536: 768 key tiles and
    768 query tiles, five or six per CTA."""
    fa = cuda_lib
    dev = torch.device("cuda", 0)
    B, H, N, d = 2, 32, 1536, 128
    q, k, v, dO = (t.to(dev) for t in _inputs(5, B, H, N, N, d))
    o, lse = fa.forward(q, k, v, causal=True)
    ws = torch.full((fa.fa_bwd_workspace_bytes(B, H, N, N, d),), 255, dtype=torch.uint8, device=dev)
    outs = []
    for _ in range(3):
        g = [torch.full_like(q, float("nan")) for _ in range(3)]
        fa.fa_bwd(q, k, v, o, lse, dO, g[0], g[1], g[2], B, H, N, N, d, d ** -0.5, True, ws, ws.numel())
        outs.append(g)
    delta = torch.empty(B, H, N, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fa.fa_bwd_preprocess(o, dO, delta, B, H, N, d)
    fa.fa_bwd_dkdv(q, k, v, lse, delta, dO, dk, dv, B, H, N, N, d, d ** -0.5, True)
    fa.fa_bwd_dq(q, k, v, lse, delta, dO, dq, B, H, N, N, d, d ** -0.5, True)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_error()[0] == 0
    for g in outs:
        assert torch.equal(g[0], dq) and torch.equal(g[1], dk) and torch.equal(g[2], dv)


# fa_bwd_dkdv_pair takes key tiles two at a time: one key tile (the odd CTA's
# tile lies wholly past Nk), odd and even tile counts, ragged and Nq != Nk.
PAIR_CASES = [
    (1, 2, 128, 128, True),
    (1, 2, 128, 128, False),
    (1, 2, 300, 300, True),
    (2, 2, 513, 257, False),
    (1, 2, 257, 513, True),
    (1, 2, 700, 200, True),
    (3, 2, 129, 129, True),
    (1, 3, 640, 384, True),
    (1, 32, 2048, 2048, True),
]


@pytest.mark.parametrize("B,H,Nq,Nk,causal", PAIR_CASES)
def test_dkdv_on_cta_pairs(cuda_lib, B, H, Nq, Nk, causal):
    """The CTA-pair dK/dV pass against the oracle, and against fa_bwd_dkdv."""
    fa = cuda_lib
    dev = torch.device("cuda", 0)
    d = 128
    scale = 1.0 / math.sqrt(d)
    q, k, v, dO = _inputs(700 + Nq + 3 * Nk + causal, B, H, Nq, Nk, d)
    qd, kd, vd, dOd = (t.to(dev) for t in (q, k, v, dO))
    o, lse = fa.forward(qd, kd, vd, scale=scale, causal=causal)
    delta = torch.empty(B, H, Nq, device=dev)
    fa.fa_bwd_preprocess(o, dOd, delta, B, H, Nq, d)
    dk, dv = torch.full_like(kd, float("nan")), torch.full_like(vd, float("nan"))
    dk1, dv1 = torch.empty_like(kd), torch.empty_like(vd)
    fa.fa_bwd_dkdv_pair(qd, kd, vd, lse, delta, dOd, dk, dv, B, H, Nq, Nk, d, scale, causal)
    fa.fa_bwd_dkdv(qd, kd, vd, lse, delta, dOd, dk1, dv1, B, H, Nq, Nk, d, scale, causal)
    torch.cuda.synchronize()
    st, detail = fa.fa_get_last_device_error()
    assert st == 0, detail
    _, rk, rv = naive.backward(f64(q), f64(k), f64(v), f64(dO), scale, causal)
    tag = "pair B%d H%d Nq%d Nk%d c%d" % (B, H, Nq, Nk, causal)
    dp_max = np.abs(f64(dO) @ np.swapaxes(f64(v), -1, -2)).max()
    cancel = scale * dp_max * np.abs(f64(q)).max()
    check_grad(f64(dk.cpu()), rk, "dK " + tag, cancel_scale=cancel)
    check_grad(f64(dv.cpu()), rv, "dV " + tag)
    # the same sums as the single-CTA pass, computed on other tensor cores: equal to
    # within fp32 accumulation order (both are rounded to bf16 at the end)
    assert (dk.float() - dk1.float()).abs().max() <= 2 ** -7 * dk1.float().abs().max() + 1e-6
    assert (dv.float() - dv1.float()).abs().max() <= 2 ** -7 * dv1.float().abs().max() + 1e-6


@pytest.mark.parametrize("N,d", [(700, 128), (300, 64)])
def test_backward_gradients_16_byte_aligned(cuda_lib, N, d):
    """dQ, dK, dV written 16 bytes past a 32-byte boundary take the 16-byte
    store path: the same bits as aligned outputs."""
    fa = cuda_lib
    dev = torch.device("cuda", 0)
    B, H = 1, 2
    q, k, v, dO = (t.to(dev) for t in _inputs(53, B, H, N, N, d))
    o, lse = fa.forward(q, k, v, causal=True)
    ref = fa.backward(q, k, v, o, lse, dO, causal=True)
    outs = []
    for _ in range(3):
        buf = torch.empty(B * H * N * d + 16, dtype=torch.bfloat16, device=dev)
        start = ((16 - buf.data_ptr() % 32) % 32) // 2
        t = buf[start:start + B * H * N * d].view(B, H, N, d)
        assert t.data_ptr() % 32 == 16
        outs.append(t)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, N, d), dtype=torch.uint8, device=dev)
    fa.fa_bwd(q, k, v, o, lse, dO, *outs, B, H, N, N, d, d ** -0.5, True, ws, ws.numel())
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_error()[0] == 0
    assert all(torch.equal(a, b) for a, b in zip(outs, ref))


def test_backward_deterministic(cuda_lib):
    """No atomics anywhere: two runs give identical bits."""
    q, k, v, dO = _inputs(9, 1, 4, 640, 640, 128)
    a = _run(cuda_lib, q, k, v, dO, 0.088, True)
    b = _run(cuda_lib, q, k, v, dO, 0.088, True)
    assert all(torch.equal(x, y) for x, y in zip(a, b))


def test_fused_backward_matches_two_pass(cuda_lib):
    """fa_bwd_fused: dK and dV are the same sums over the same query tiles as
    fa_bwd's, in 64-row instead of 128-row tiles; dQ differs only in the order
    of its fp32 additions.  All three agree with fa_bwd to within bf16 rounding,
    and dK, dV repeat bit for bit from run to run."""
    q, k, v, dO = _inputs(19, 1, 4, 1000, 1000, 128)
    ref = _run(cuda_lib, q, k, v, dO, 0.088, True)
    a = _run(cuda_lib, q, k, v, dO, 0.088, True, fused=True)
    b = _run(cuda_lib, q, k, v, dO, 0.088, True, fused=True)
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    for x, y in zip(a, ref):
        assert (x.float() - y.float()).abs().max() <= 2 ** -7 * y.float().abs().max() + 1e-6


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("N", [1024, 2048, 4096, 8192])
def test_backward_full_size_sweep(cuda_lib, N, fused):
    """B=1, H=32, d=128, causal, N in the 1k-8k sweep: heads 0 and 31 against the
    oracle, for fa_bwd and for fa_bwd_fused."""
    cfg = syn.CONFIGS["fwd_bwd_sweep"]
    B, H, d = cfg["B"], cfg["H"], cfg["d"]
    seed = cfg["seed"] + N
    q, k, v, dO = _inputs(seed, B, H, N, N, d)
    scale = syn.default_scale(d)
    dq, dk, dv = _run(cuda_lib, q, k, v, dO, scale, True, fused)
    for h in (0, H - 1):
        rq, rk, rv = naive.backward(f64(q[0, h]), f64(k[0, h]), f64(v[0, h]), f64(dO[0, h]), scale, True)
        check_grad(f64(dq[0, h]), rq, "dQ N%d h%d" % (N, h))
        check_grad(f64(dk[0, h]), rk, "dK N%d h%d" % (N, h))
        check_grad(f64(dv[0, h]), rv, "dV N%d h%d" % (N, h))
    for g in (dq, dk, dv):
        assert torch.isfinite(g.float()).all()


def test_forward_backward_in_cuda_graph(cuda_lib):
    """fa_fwd and fa_bwd (with its programmatic dependent launches) captured in a
    CUDA graph and replayed give the eager results bit for bit."""
    fa = cuda_lib
    dev = torch.device("cuda", 0)
    B, H, N, d = 1, 8, 1024, 128
    q, k, v, dO = (t.to(dev) for t in _inputs(77, B, H, N, N, d))
    o, lse = torch.empty_like(q), torch.empty(B, H, N, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, N, d), dtype=torch.uint8, device=dev)

    def step():
        fa.fa_fwd(q, k, v, o, lse, B, H, N, N, d, d ** -0.5, True)
        fa.fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, N, d, d ** -0.5, True, ws, ws.numel())

    step()
    torch.cuda.synchronize()
    ref = [t.clone() for t in (o, lse, dq, dk, dv)]
    for t in (o, lse, dq, dk, dv):
        t.fill_(float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # warm-up on the side stream before capture
    torch.cuda.current_stream().wait_stream(s)
    for t in (o, lse, dq, dk, dv):
        t.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    g.replay()
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_error()[0] == 0
    for a, b in zip(ref, (o, lse, dq, dk, dv)):
        assert torch.equal(a, b)


def test_forward_backward_past_32_bit_offsets(cuda_lib):
    """B=1, H=4096, N=4096, d=128, causal: each of Q, K, V, O, dO and the three
    gradients holds 2^31 elements, so element offsets need more than 31 bits.
    Inputs are drawn on the device; heads 0 and 4095 (the last rows of every
    tensor) against the oracle, forward and backward."""
    fa = cuda_lib
    dev = torch.device("cuda", 0)
    B, H, N, d = 1, 4096, 4096, 128
    g = torch.Generator(device=dev).manual_seed(4096)
    q, k, v, dO = (torch.empty(B, H, N, d, dtype=torch.bfloat16, device=dev).normal_(generator=g) for _ in range(4))
    o, lse = fa.forward(q, k, v, causal=True)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, N, d), dtype=torch.uint8, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fa.fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, N, d, d ** -0.5, True, ws, ws.numel())
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_error()[0] == 0
    for h in (0, H - 1):
        sl = slice(h, h + 1)
        qh, kh, vh, dOh = (f64(t[:, sl].cpu()) for t in (q, k, v, dO))
        o_ref, lse_ref = naive.forward(qh, kh, vh, d ** -0.5, True)
        check_out(f64(o[:, sl].cpu()), f64(lse[:, sl].cpu()), o_ref, lse_ref, "O, LSE head %d" % h)
        rq, rk, rv = naive.backward(qh, kh, vh, dOh, d ** -0.5, True)
        check_grad(f64(dq[:, sl].cpu()), rq, "dQ head %d" % h)
        check_grad(f64(dk[:, sl].cpu()), rk, "dK head %d" % h)
        check_grad(f64(dv[:, sl].cpu()), rv, "dV head %d" % h)


def _bits(t):
    return t.view(torch.int16 if t.element_size() == 2 else torch.int32)


@pytest.mark.parametrize("N", [1024, 2048])
def test_repeated_runs_repeat_bits(cuda_lib, N):
    """Many back-to-back calls at B=1, H=32, d=128, causal, each compared bit for bit
    with the first: the forward (O, LSE), fa_bwd (dQ, dK, dV), fa_bwd_fused (dK, dV;
    its dQ adds in a run-dependent order) and fa_bwd_dkdv_pair (dK, dV).  Every result
    is a fixed sum in a fixed order, so a hand-off between warps that let a product
    read a tile before all of it was written shows up as changed bits."""
    fa = cuda_lib
    dev = torch.device("cuda", 0)
    B, H, d, reps = 1, 32, 128, 25
    scale = syn.default_scale(d)
    q, k, v, dO = (t.to(dev) for t in _inputs(31 + N, B, H, N, N, d))
    o0, lse0 = fa.forward(q, k, v, scale=scale, causal=True)
    ref_bwd = fa.backward(q, k, v, o0, lse0, dO, scale=scale, causal=True)
    ref_fused = fa.backward(q, k, v, o0, lse0, dO, scale=scale, causal=True, fused=True)[1:]
    delta = torch.empty(B, H, N, device=dev)
    fa.fa_bwd_preprocess(o0, dO, delta, B, H, N, d)
    ref_pair = (torch.empty_like(k), torch.empty_like(v))
    fa.fa_bwd_dkdv_pair(q, k, v, lse0, delta, dO, *ref_pair, B, H, N, N, d, scale, True)
    same = torch.ones((), dtype=torch.bool, device=dev)
    for _ in range(reps):
        o, lse = fa.forward(q, k, v, scale=scale, causal=True)
        g = fa.backward(q, k, v, o0, lse0, dO, scale=scale, causal=True)
        gf = fa.backward(q, k, v, o0, lse0, dO, scale=scale, causal=True, fused=True)[1:]
        gp = (torch.empty_like(k), torch.empty_like(v))
        fa.fa_bwd_dkdv_pair(q, k, v, lse0, delta, dO, *gp, B, H, N, N, d, scale, True)
        for x, y in zip((o, lse) + tuple(g) + tuple(gf) + gp, (o0, lse0) + tuple(ref_bwd) + tuple(ref_fused) + ref_pair):
            same &= (_bits(x) == _bits(y)).all()  # on the device: the calls stay back to back
    torch.cuda.synchronize()
    st, detail = fa.fa_get_last_device_error()
    assert st == 0, detail
    assert bool(same)
    for x in (o0,) + tuple(ref_bwd):
        assert torch.isfinite(x.float()).all()
