"""Forward parity: the CUDA path (through the C ABI) against the fp64 oracle,
element by element, on the same seeded bf16 inputs."""
import math

import numpy as np
import pytest
import torch

from exact_tiled_attention_21_gb300 import synthetic as syn
from oracle import naive
from tests.parity import check_out, derived_o_bound, f64

pytestmark = pytest.mark.gpu


def _inputs(seed, B, H, Nq, Nk, d, std=1.0):
    q = syn.bhnd(seed, syn.TAG_Q, B, H, Nq, d, std)
    k = syn.bhnd(seed, syn.TAG_K, B, H, Nk, d, std)
    v = syn.bhnd(seed, syn.TAG_V, B, H, Nk, d, std)
    return q, k, v


def _run(fa, q, k, v, scale, causal):
    dev = torch.device("cuda", 0)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o, lse = fa.forward(qd, kd, vd, scale=scale, causal=causal)
    torch.cuda.synchronize()
    st, detail = fa.fa_get_last_device_error()
    assert st == 0, detail
    return o.cpu(), lse.cpu()


# (B, H, Nq, Nk, d, causal): several tiles, ragged tails, Nq != Nk both ways,
# rows that see no key, single rows and single keys.
CASES = [
    (1, 2, 128, 128, 64, False),     # the small workload
    (1, 2, 128, 128, 64, True),
    (1, 3, 300, 300, 64, True),
    (1, 2, 1000, 1000, 128, False),
    (1, 2, 1000, 1000, 128, True),
    (2, 2, 513, 257, 128, False),
    (2, 2, 257, 513, 64, False),
    (1, 2, 200, 700, 128, True),     # queries see a prefix of 500 + i keys
    (1, 2, 700, 200, 128, True),     # the first 500 queries see no key
    (1, 2, 700, 200, 64, True),
    (1, 1, 1, 1, 64, False),
    (1, 1, 1, 1, 128, True),
    (1, 2, 1, 5000, 128, False),
    (1, 2, 5000, 1, 64, False),
    (2, 3, 77, 1031, 64, True),
    (1, 1, 2048, 2048, 128, True),
]


def test_forward_cases_cover_split_tiles(cuda_lib):
    """Most small cases above run through split-KV tiles (odd and even key
    block counts, ragged tails, rows that see no key); single-tile ones through
    256-row tiles."""
    rows = [cuda_lib.fa_fwd_tile_rows(B, H, Nq, Nk, d, c) for B, H, Nq, Nk, d, c in CASES]
    assert rows.count(128) >= 10 and rows.count(256) >= 2, rows


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", CASES)
def test_forward_parity(cuda_lib, B, H, Nq, Nk, d, causal):
    seed = 100 + Nq * 7 + Nk + d + causal
    q, k, v = _inputs(seed, B, H, Nq, Nk, d)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(cuda_lib, q, k, v, scale, causal)
    o_ref, lse_ref = naive.forward(f64(q), f64(k), f64(v), scale, causal)
    check_out(f64(o), f64(lse), o_ref, lse_ref, "B%d H%d Nq%d Nk%d d%d c%d" % (B, H, Nq, Nk, d, causal))


# Enough heads for the 256-row tiles (two query tiles per CTA); most cases
# above take split-KV tiles.
WIDE_CASES = [
    (2, 80, 513, 600, 64, True),
    (4, 40, 700, 200, 64, True),     # rows that see no key
    (4, 80, 300, 777, 128, False),
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", WIDE_CASES)
def test_forward_parity_256_row_tiles(cuda_lib, B, H, Nq, Nk, d, causal):
    assert cuda_lib.fa_fwd_tile_rows(B, H, Nq, Nk, d, causal) == 256
    seed = 300 + Nq * 7 + Nk + d + causal
    q, k, v = _inputs(seed, B, H, Nq, Nk, d)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(cuda_lib, q, k, v, scale, causal)
    o_ref, lse_ref = naive.forward(f64(q), f64(k), f64(v), scale, causal)
    check_out(f64(o), f64(lse), o_ref, lse_ref, "B%d H%d Nq%d Nk%d d%d c%d" % (B, H, Nq, Nk, d, causal))


def test_forward_tile_modes_agree(cuda_lib):
    """The same heads through split-KV tiles (a batch of 2 heads) and through
    256-row tiles (those heads inside a batch of 320): the two orders of the
    online recurrence agree within the bf16 output's rounding."""
    B, H, N, d = 1, 320, 768, 64
    for causal in (False, True):
        assert cuda_lib.fa_fwd_tile_rows(B, H, N, N, d, causal) == 256
        assert cuda_lib.fa_fwd_tile_rows(1, 2, N, N, d, causal) == 128
    q, k, v = _inputs(41, B, H, N, N, d)
    for causal in (False, True):
        o_wide, l_wide = _run(cuda_lib, q, k, v, 0.125, causal)
        o_split, l_split = _run(cuda_lib, q[:, :2].contiguous(), k[:, :2].contiguous(), v[:, :2].contiguous(),
                                0.125, causal)
        assert (o_wide[:, :2].float() - o_split.float()).abs().max() <= 2 ** -7
        assert (l_wide[:, :2] - l_split).abs().max() <= 1e-4


def _offset16(shape, dtype, dev):
    """A contiguous tensor whose data starts 16 bytes past a 32-byte boundary
    (the C ABI asks for 16-byte alignment only)."""
    elems = 16 // torch.empty(0, dtype=dtype).element_size()
    n = int(np.prod(shape))
    buf = torch.empty(n + 2 * elems, dtype=dtype, device=dev)
    base = buf.data_ptr() % 32
    start = ((16 - base) % 32) // buf.element_size()
    t = buf[start:start + n].view(*shape)
    assert t.data_ptr() % 32 == 16
    return t


@pytest.mark.parametrize("B,H,N,d,causal", [(1, 2, 300, 128, True), (1, 2, 700, 64, False), (1, 320, 768, 64, True)])
def test_forward_output_16_byte_aligned(cuda_lib, B, H, N, d, causal):
    """O written at an address that is 16- but not 32-byte aligned takes the
    16-byte store path: the same bits as an aligned O, in both tile modes."""
    fa = cuda_lib
    dev = torch.device("cuda", 0)
    q, k, v = (t.to(dev) for t in _inputs(47, B, H, N, N, d))
    o_ref, lse_ref = fa.forward(q, k, v, causal=causal)
    o = _offset16((B, H, N, d), torch.bfloat16, dev)
    lse = torch.empty(B, H, N, device=dev)
    fa.fa_fwd(q, k, v, o, lse, B, H, N, N, d, d ** -0.5, causal)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_error()[0] == 0
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


def test_forward_scale_argument(cuda_lib):
    """A non-default scale reaches the kernel (LSE shifts with it).  Off the
    workloads' scale the max-abs bound is the one derived from the two bf16
    roundings (tests/parity.py), not the workloads' fixed 1e-2."""
    q, k, v = _inputs(7, 1, 2, 256, 384, 128)
    for scale in (0.02, 0.3):
        o, lse = _run(cuda_lib, q, k, v, scale, False)
        o_ref, lse_ref = naive.forward(f64(q), f64(k), f64(v), scale, False)
        check_out(f64(o), f64(lse), o_ref, lse_ref, "scale %g" % scale,
                  max_abs=derived_o_bound(f64(v)))


@pytest.mark.parametrize("causal", [False, True])
def test_forward_growing_scores(cuda_lib, causal):
    """Key rows scaled by a ramp (0.5 at the first key to 12.5 at the last): the
    row max keeps growing from key block to key block, by more than 2^8 in the
    log2 domain every block or two, so the accumulator is rescaled over and
    over (the lazy-rescale path).  Off the workloads' scores, so the max-abs
    bound is the one derived from the bf16 roundings."""
    B, H, N, d = 1, 2, 1024, 128
    q, k, v = _inputs(61, B, H, N, N, d)
    ramp = 0.5 + 12.0 * torch.arange(N, dtype=torch.float32) / N
    k = (k.float() * ramp[None, None, :, None]).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(cuda_lib, q, k, v, scale, causal)
    o_ref, lse_ref = naive.forward(f64(q), f64(k), f64(v), scale, causal)
    check_out(f64(o), f64(lse), o_ref, lse_ref, "growing scores causal%d" % causal, max_abs=derived_o_bound(f64(v)))


def test_forward_repeatable(cuda_lib):
    """The forward has no atomics: two runs are bitwise identical."""
    q, k, v = _inputs(8, 1, 4, 640, 640, 128)
    o1, l1 = _run(cuda_lib, q, k, v, 0.088, True)
    o2, l2 = _run(cuda_lib, q, k, v, 0.088, True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("causal", [False, True])
def test_forward_full_size_4k(cuda_lib, causal):
    """B=2, H=32, N=4096, d=128: every head of batch 0 against the oracle."""
    cfg = syn.CONFIGS["fwd_4k"]
    B, H, N, d = cfg["B"], cfg["H"], cfg["Nq"], cfg["d"]
    q, k, v = _inputs(cfg["seed"], B, H, N, N, d)
    scale = syn.default_scale(d)
    o, lse = _run(cuda_lib, q, k, v, scale, causal)
    for h in range(H):
        o_ref, lse_ref = naive.forward(f64(q[0, h]), f64(k[0, h]), f64(v[0, h]), scale, causal)
        check_out(f64(o[0, h]), f64(lse[0, h]), o_ref, lse_ref, "head %d" % h)
    assert torch.isfinite(o[1].float()).all() and torch.isfinite(lse[1]).all()


def test_forward_long_context(cuda_lib):
    """B=1, H=32, N=131072, d=128, causal, N(0, 0.5^2): 256 seeded rows over 4
    heads against the oracle, and no N x N buffer (peak memory near Q,K,V,O,LSE)."""
    cfg = syn.CONFIGS["long_causal"]
    B, H, N, d = cfg["B"], cfg["H"], cfg["Nq"], cfg["d"]
    dev = torch.device("cuda", 0)
    torch.cuda.reset_peak_memory_stats(dev)
    base = torch.cuda.memory_allocated(dev)
    qd = syn.bhnd(cfg["seed"], syn.TAG_Q, B, H, N, d, cfg["std"]).to(dev)
    kd = syn.bhnd(cfg["seed"], syn.TAG_K, B, H, N, d, cfg["std"]).to(dev)
    vd = syn.bhnd(cfg["seed"], syn.TAG_V, B, H, N, d, cfg["std"]).to(dev)
    o, lse = cuda_lib.forward(qd, kd, vd, causal=True)
    torch.cuda.synchronize()
    st, detail = cuda_lib.fa_get_last_device_error()
    assert st == 0, detail
    peak = torch.cuda.max_memory_allocated(dev) - base
    floor = 4 * B * H * N * d * 2 + B * H * N * 4
    assert peak <= floor * 1.01 + (64 << 20), (peak, floor)
    scale = syn.default_scale(d)
    heads = syn.sample_heads(cfg["seed"], H, cfg["sample_heads"])
    for h in heads:
        rows = syn.sample_rows(cfg["seed"] * 1000 + h, N, cfg["sample_rows"], must=(0,))
        q_rows = qd[0, h, rows].cpu()
        o_ref, lse_ref = naive.forward(f64(q_rows), f64(kd[0, h].cpu()), f64(vd[0, h].cpu()), scale,
                                       True, rows=rows, Nq=N)
        check_out(f64(o[0, h, rows].cpu()), f64(lse[0, h, rows].cpu()), o_ref, lse_ref, "head %d" % h)
