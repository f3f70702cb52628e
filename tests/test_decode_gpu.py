"""Split-KV decode parity against the fp64 oracle (through the C ABI)."""
import math

import pytest
import torch

from exact_tiled_attention_21_gb300 import synthetic as syn
from oracle import naive
from tests.parity import check_out, f64

pytestmark = pytest.mark.gpu


def _inputs(seed, B, H, Nk, d):
    q = syn.bhd(seed, syn.TAG_Q, B, H, d)
    kc = syn.bhnd(seed, syn.TAG_K, B, H, Nk, d)
    vc = syn.bhnd(seed, syn.TAG_V, B, H, Nk, d)
    return q, kc, vc


def _run(fa, q, kc, vc, scale, splits):
    dev = torch.device("cuda", 0)
    o, lse = fa.decode(q.to(dev), kc.to(dev), vc.to(dev), scale=scale, num_splits=splits)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


# (B, H, Nk, d, splits): chunks of several 128-key pieces, ragged chunks,
# empty trailing splits (Nk < splits), a single key, automatic split count.
# d = 128 with Nk a multiple of 128 runs on the tensor-core kernel (whole
# 128-key stages per split, so trailing splits can be empty there too); every
# other shape on the 16-byte-load kernel.  B=8 H=32 and B=16 H=32 let the
# automatic count of that kernel fall below its length cap (several hundred
# heads: it keeps the (b, h, split) grid within whole waves of resident CTAs);
# B=2100 has more sequences than the tensor-core kernel stages lengths for.
CASES = [
    (1, 2, 128, 128, 1),
    (2, 3, 256, 128, 16),
    (3, 2, 384, 128, 0),
    (2, 2, 8192, 128, 7),
    (2, 3, 4096, 128, 16),
    (2, 3, 1000, 128, 16),
    (1, 4, 37, 128, 16),
    (1, 2, 5, 64, 16),
    (1, 1, 1, 128, 1),
    (3, 2, 2000, 64, 3),
    (1, 2, 5000, 64, 0),
    (1, 2, 70000, 128, 0),
    (1, 1, 777, 128, 256),
    (2, 3, 4001, 128, 16),
    (1, 2, 129, 128, 4),
    (2, 3, 4096, 64, 16),
    (2, 2, 1000, 64, 0),
    (1, 1, 777, 64, 256),
    (1, 2, 64, 64, 4),
    (1, 2, 8, 128, 1),
    (1, 2, 100, 128, 4),
    (2, 3, 70000, 64, 0),
    (8, 32, 4000, 128, 0),
    (16, 32, 2048, 64, 0),
    (2100, 2, 256, 128, 0),
]


@pytest.mark.parametrize("B,H,Nk,d,splits", CASES)
def test_decode_parity(cuda_lib, B, H, Nk, d, splits):
    q, kc, vc = _inputs(300 + Nk + d, B, H, Nk, d)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(cuda_lib, q, kc, vc, scale, splits)
    o_ref, lse_ref = naive.decode(f64(q), f64(kc), f64(vc), scale)
    check_out(f64(o), f64(lse), o_ref, lse_ref, "B%d H%d Nk%d d%d S%d" % (B, H, Nk, d, splits))


def test_decode_full_size(cuda_lib):
    """B=32, H=32, Nk=4096, d=128, 16 splits: every (b, h) against the oracle."""
    cfg = syn.CONFIGS["decode"]
    B, H, Nk, d = cfg["B"], cfg["H"], cfg["Nk"], cfg["d"]
    q, kc, vc = _inputs(cfg["seed"], B, H, Nk, d)
    scale = syn.default_scale(d)
    o, lse = _run(cuda_lib, q, kc, vc, scale, cfg["splits"])
    o_ref, lse_ref = naive.decode(f64(q), f64(kc), f64(vc), scale)
    check_out(f64(o), f64(lse), o_ref, lse_ref, "decode full")


def test_decode_without_lse(cuda_lib):
    q, kc, vc = _inputs(5, 1, 2, 300, 128)
    dev = torch.device("cuda", 0)
    o = cuda_lib.decode(q.to(dev), kc.to(dev), vc.to(dev), num_splits=4, want_lse=False)
    o_ref, _ = naive.decode(f64(q), f64(kc), f64(vc), 1 / math.sqrt(128))
    check_out(f64(o.cpu()), None, o_ref, None, "no lse")


@pytest.mark.parametrize("d", [128, 64])
def test_decode_caches_past_32_bit_offsets(cuda_lib, d):
    """H=64, Nk=128 and B=4096 (d=128, the tensor-core kernel) or B=8192 (d=64, the
    16-byte-load kernel): each cache holds 2^32 elements, so element offsets need
    64 bits.  The caches are drawn on the device; 64 (b, h) rows spread over the
    whole range, the last one included, against the oracle."""
    dev = torch.device("cuda", 0)
    B, H, Nk = (4096 if d == 128 else 8192), 64, 128
    g = torch.Generator(device=dev).manual_seed(2 ** 31 + d)
    q = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev).normal_(generator=g)
    kc = torch.empty(B, H, Nk, d, dtype=torch.bfloat16, device=dev).normal_(generator=g)
    vc = torch.empty(B, H, Nk, d, dtype=torch.bfloat16, device=dev).normal_(generator=g)
    o, lse = cuda_lib.decode(q, kc, vc, num_splits=0)
    torch.cuda.synchronize()
    idx = torch.linspace(0, B * H - 1, 64).round().long()
    b, h = idx // H, idx % H
    o_s, lse_s = o[b, h].cpu()[None], lse[b, h].cpu()[None]
    q_s, k_s, v_s = q[b, h].cpu()[None], kc[b, h].cpu()[None], vc[b, h].cpu()[None]
    del kc, vc
    o_ref, lse_ref = naive.decode(f64(q_s), f64(k_s), f64(v_s), 1 / math.sqrt(d))
    check_out(f64(o_s), f64(lse_s), o_ref, lse_ref, "2^32-element caches d%d" % d)


@pytest.mark.parametrize("Nk,d,splits", [(4096, 128, 16), (4000, 128, 0), (4096, 64, 0)])
def test_decode_repeats_bits(cuda_lib, Nk, d, splits):
    """B=32, H=32: 50 back-to-back calls give the first call's O and LSE bit for
    bit (the splits' partials are combined in a fixed order; no atomics)."""
    fa = cuda_lib
    dev = torch.device("cuda", 0)
    q, kc, vc = (t.to(dev) for t in _inputs(40 + Nk + d, 32, 32, Nk, d))
    o0, lse0 = fa.decode(q, kc, vc, num_splits=splits)
    same = torch.ones((), dtype=torch.bool, device=dev)
    for _ in range(50):
        o, lse = fa.decode(q, kc, vc, num_splits=splits)
        same &= (o.view(torch.int16) == o0.view(torch.int16)).all()
        same &= (lse.view(torch.int32) == lse0.view(torch.int32)).all()
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_error()[0] == 0
    assert bool(same)
