"""Paged, grouped-query decode (fa_decode_paged) against the fp64 oracle
(oracle.naive.decode_paged: the plain decode of each query head against its
sequence's tokens gathered through the block table)."""
import math

import numpy as np
import pytest
import torch

import exact_tiled_attention_21_gb300 as fa_mod
from exact_tiled_attention_21_gb300 import synthetic as syn
from oracle import naive
from tests.parity import check_out, check_out_elementwise, f64

pytestmark = pytest.mark.gpu


def _case(seed, B, Hq, Hkv, P, lens, d, extra_pages=5):
    rng = np.random.default_rng(seed)
    maxp = max(-(-L // P) for L in lens)
    npages = B * maxp + extra_pages
    q = syn.bhd(seed, syn.TAG_Q, B, Hq, d)
    kp = syn.bhnd(seed, syn.TAG_K, npages, Hkv, P, d)   # [num_pages, Hkv, P, d]
    vp = syn.bhnd(seed, syn.TAG_V, npages, Hkv, P, d)
    table = rng.permutation(npages)[:B * maxp].reshape(B, maxp).astype(np.int32)
    return q, kp, vp, table, np.array(lens, dtype=np.int32)


def _run(fa, q, kp, vp, table, lens, splits):
    dev = torch.device("cuda", 0)
    o, lse = fa.decode_paged(q.to(dev), kp.to(dev), vp.to(dev), torch.from_numpy(table).to(dev),
                             torch.from_numpy(lens).to(dev), num_splits=splits)
    torch.cuda.synchronize()
    st, detail = fa.fa_get_last_device_error()
    assert st == 0, detail
    return o.cpu(), lse.cpu()


# (B, Hq, Hkv, page, lens, d, splits)
CASES = [
    (3, 8, 2, 16, [1, 37, 200], 128, 4),        # group of 4
    (2, 6, 2, 64, [64, 1000], 64, 16),          # group of 3 (one head per CTA)
    (2, 16, 2, 32, [4096, 513], 128, 16),       # group of 8 (two CTAs per kv head)
    (2, 8, 1, 16, [300, 17], 128, 8),           # multi-query (one kv head)
    (2, 4, 4, 8, [129, 1], 64, 3),              # one query head per kv head
    (1, 4, 2, 1, [77], 128, 16),                # single-token pages
    (2, 4, 2, 16, [5, 3], 128, 16),             # more splits than tokens: empty splits
    (2, 32, 2, 8, [1000, 129], 128, 5),         # 8-token pages, group of 16 (one full MMA group)
    (2, 8, 2, 128, [700, 128], 128, 3),         # one page per 128-key stage
    (2, 8, 2, 256, [1000, 300], 128, 2),        # pages longer than a stage
    (1, 32, 1, 16, [517], 128, 4),              # multi-query, 32 heads: two groups of 16
    (1, 40, 2, 32, [333], 128, 2),              # group of 20: 16 + 4 heads
    (1, 8, 2, 48, [500], 128, 3),               # 48-token pages (not a divisor of 128): boxes of 16 rows
    (2, 8, 2, 40, [1000, 41], 128, 3),          # 40-token pages: boxes of 8 rows, 16 per stage
    (2, 16, 4, 24, [777, 24], 128, 0),          # 24-token pages, automatic split count
    (2, 8, 2, 80, [1000, 79], 128, 4),          # 80-token pages: boxes of 16 rows
    (2, 8, 2, 96, [1100, 97], 64, 3),           # d = 64, 96-token pages: boxes of 32 rows
    (2, 8, 2, 136, [1000, 136], 128, 2),        # pages longer than a stage, boxes of 8 rows
    (2, 8, 2, 160, [1000, 161], 128, 3),        # pages longer than a stage, boxes of 32 rows
    (2, 16, 4, 192, [900, 385], 128, 0),        # boxes of 64 rows, automatic split count
    (2, 8, 2, 200, [1500, 199], 64, 2),         # d = 64, pages longer than a stage, boxes of 8 rows
    (1, 8, 2, 16, [20000], 128, 1),             # one split: 157 stages through the ring
    (32, 32, 8, 16, [4096] * 30 + [1, 777], 128, 0),  # automatic split count (tensor-core path)
    (3, 8, 2, 48, [1000, 3, 480], 128, 0),      # automatic split count, 48-token pages
    (3, 8, 2, 20, [1000, 3, 480], 128, 0),      # automatic split count (general path: 20-token pages)
    (2, 8, 2, 12, [500, 77], 128, 3),           # general path, group of 4
    (2, 32, 2, 8, [1000, 129], 64, 5),          # d = 64 on the tensor cores: 8-token pages, group of 16
    (2, 8, 2, 256, [1000, 300], 64, 2),         # d = 64, pages longer than a stage
    (1, 40, 2, 32, [333], 64, 2),               # d = 64, group of 20
    (1, 8, 2, 16, [20000], 64, 1),              # d = 64, 157 stages through the ring
    (32, 32, 8, 16, [4096] * 30 + [1, 777], 64, 0),  # d = 64, automatic split count
    (2, 8, 2, 48, [500, 77], 64, 3),            # d = 64, 48-token pages
    (2, 8, 2, 20, [500, 77], 64, 3),            # d = 64, general path (20-token pages)
]


@pytest.mark.parametrize("B,Hq,Hkv,P,lens,d,splits", CASES)
def test_paged_decode_parity(cuda_lib, B, Hq, Hkv, P, lens, d, splits):
    q, kp, vp, table, L = _case(900 + P + d + Hq, B, Hq, Hkv, P, lens, d)
    o, lse = _run(cuda_lib, q, kp, vp, table, L, splits)
    o_ref, lse_ref = naive.decode_paged(f64(q), f64(kp), f64(vp), table, L, 1 / math.sqrt(d))
    check_out(f64(o), f64(lse), o_ref, lse_ref, "B%d Hq%d Hkv%d P%d d%d" % (B, Hq, Hkv, P, d))


def test_paged_decode_full_size(cuda_lib):
    """B=32, Hq=32, Hkv=8 (groups of 4), 16-token pages, lengths up to 4096."""
    rng = np.random.default_rng(77)
    lens = [4096, 1] + list(rng.integers(1, 4097, size=30))
    q, kp, vp, table, L = _case(78, 32, 32, 8, 16, lens, 128)
    o, lse = _run(cuda_lib, q, kp, vp, table, L, 16)
    o_ref, lse_ref = naive.decode_paged(f64(q), f64(kp), f64(vp), table, L, 1 / math.sqrt(128))
    check_out(f64(o), f64(lse), o_ref, lse_ref, "paged full size")


def test_paged_decode_matches_contiguous_decode(cuda_lib):
    """Identity table, full lengths, Hq == Hkv: the same as fa_decode."""
    B, H, P, npg, d = 2, 4, 64, 8, 128
    q = syn.bhd(5, syn.TAG_Q, B, H, d)
    kc, vc = syn.bhnd(5, syn.TAG_K, B, H, P * npg, d), syn.bhnd(5, syn.TAG_V, B, H, P * npg, d)
    kp = kc.reshape(B, H, npg, P, d).permute(0, 2, 1, 3, 4).reshape(B * npg, H, P, d).contiguous()
    vp = vc.reshape(B, H, npg, P, d).permute(0, 2, 1, 3, 4).reshape(B * npg, H, P, d).contiguous()
    table = np.arange(B * npg, dtype=np.int32).reshape(B, npg)
    o, lse = _run(cuda_lib, q, kp, vp, table, np.full(B, P * npg, dtype=np.int32), 16)
    dev = torch.device("cuda", 0)
    o2, lse2 = cuda_lib.decode(q.to(dev), kc.to(dev), vc.to(dev), num_splits=16)
    check_out(f64(o), f64(lse), f64(o2.cpu()), f64(lse2.cpu()), "paged vs contiguous")


def test_paged_decode_rejects_bad_page_index_on_device(cuda_lib):
    """A page index outside the cache is never dereferenced: it reads as zeros
    and the kernel records FA_ERR_INVALID_ARG."""
    q, kp, vp, table, L = _case(5, 1, 4, 2, 16, [40], 128)
    table[0, 1] = kp.shape[0] + 1000
    dev = torch.device("cuda", 0)
    cuda_lib.decode_paged(q.to(dev), kp.to(dev), vp.to(dev), torch.from_numpy(table).to(dev),
                          torch.from_numpy(L).to(dev), num_splits=4)
    st, detail = cuda_lib.fa_get_last_device_error()
    assert st == fa_mod.FA_ERR_INVALID_ARG, detail
    assert cuda_lib.fa_get_last_device_error()[0] == 0


@pytest.mark.parametrize("P,d", [(16, 128), (48, 128), (256, 128), (20, 128), (16, 64), (48, 64), (256, 64)])
def test_paged_decode_ignores_unused_slots(cuda_lib, P, d):
    """Tokens past seq_lens[b] in the last page, and pages no table names,
    may hold anything (NaN here): the result depends only on the tokens in
    range."""
    lens = [P * 3 + 5, 1, 2 * P]
    q, kp, vp, table, L = _case(31 + P, 3, 8, 2, P, lens, d)
    kp_bad, vp_bad = kp.clone(), vp.clone()
    used = np.zeros((kp.shape[0], P), dtype=bool)
    for b, n in enumerate(lens):
        for t in range(n):
            used[table[b, t // P], t % P] = True
    mask = torch.from_numpy(~used)[:, None, :, None].expand_as(kp)
    kp_bad[mask] = float("nan")
    vp_bad[mask] = float("nan")
    o, lse = _run(cuda_lib, q, kp_bad, vp_bad, table, L, 4)
    o_ref, lse_ref = naive.decode_paged(f64(q), f64(kp), f64(vp), table, L, 1 / math.sqrt(d))
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    check_out(f64(o), f64(lse), o_ref, lse_ref, "unused slots P%d d%d" % (P, d))


@pytest.mark.parametrize("d", [128, 64])
def test_paged_decode_growing_scores(cuda_lib, d):
    """Key norms that grow along the sequence raise every head's running
    maximum by far more than 2^8 between stages, so the output accumulator
    is rescaled many times within one split."""
    B, Hq, Hkv, P, n = 1, 8, 2, 16, 3000
    q, kp, vp, table, L = _case(44, B, Hq, Hkv, P, [n], d)
    ramp = torch.zeros(kp.shape[0], 1, P, 1)
    for t in range(n):
        ramp[table[0, t // P], 0, t % P, 0] = 0.5 + 12.0 * t / n
    kp = (kp.float() * ramp).to(torch.bfloat16)
    o, lse = _run(cuda_lib, q, kp, vp, table, L, 1)
    o_ref, lse_ref = naive.decode_paged(f64(q), f64(kp), f64(vp), table, L, 1 / math.sqrt(d))
    # late keys dominate (|O| ~ |v|): the rounding bound per element applies
    vmax = float(np.abs(f64(vp)).max())
    check_out_elementwise(f64(o), f64(lse), o_ref, lse_ref, vmax, "growing scores")


@pytest.mark.parametrize("d,splits", [(128, 0), (64, 3)])
def test_paged_decode_more_sequences_than_staged_lengths(cuda_lib, d, splits):
    """B=2100 sequences on the tensor-core path: the kernel stages the first
    2048 lengths in shared memory and reads the others per work item.  Every
    sequence against the oracle (lengths 1..200, 16-token pages, groups of 4)."""
    rng = np.random.default_rng(2100 + d)
    lens = list(rng.integers(1, 201, size=2100))
    lens[2047], lens[2048], lens[2099] = 200, 1, 129  # either side of the staged range
    q, kp, vp, table, L = _case(61 + d, 2100, 8, 2, 16, lens, d)
    o, lse = _run(cuda_lib, q, kp, vp, table, L, splits)
    o_ref, lse_ref = naive.decode_paged(f64(q), f64(kp), f64(vp), table, L, 1 / math.sqrt(d))
    check_out(f64(o), f64(lse), o_ref, lse_ref, "B2100 d%d" % d)


def test_paged_decode_length_out_of_range_past_the_staged_lengths(cuda_lib):
    """A length above max_pages * page for a sequence past the first 2048 is
    clamped to the table, never read past it, and recorded as
    FA_ERR_INVALID_ARG; the other sequences are unaffected."""
    lens = [40] * 2060
    q, kp, vp, table, L = _case(8, 2060, 4, 2, 16, lens, 128)
    L[2050] = 10 ** 6
    dev = torch.device("cuda", 0)
    o, lse = cuda_lib.decode_paged(q.to(dev), kp.to(dev), vp.to(dev), torch.from_numpy(table).to(dev),
                                   torch.from_numpy(L).to(dev), num_splits=2)
    st, detail = cuda_lib.fa_get_last_device_error()
    assert st == fa_mod.FA_ERR_INVALID_ARG, detail
    assert detail[2] == 2050 and detail[3] == 10 ** 6
    L_ok = L.copy()
    L_ok[2050] = table.shape[1] * 16  # the clamped length: the whole table row
    o_ref, lse_ref = naive.decode_paged(f64(q), f64(kp), f64(vp), table, L_ok, 1 / math.sqrt(128))
    check_out(f64(o.cpu()), f64(lse.cpu()), o_ref, lse_ref, "clamped length")


@pytest.mark.parametrize("P", [16, 48, 20])
def test_paged_decode_cache_past_32_bit_offsets(cuda_lib, P):
    """B=64 sequences, Hq=32, Hkv=8, d=128, pages scattered in a random order over a
    pool of 2^31 elements per cache, so page offsets need 64 bits (16- and 48-token
    pages on the tensor-core kernel, 20-token pages on the general one).  Three sequences,
    one of them short, against the oracle on their own pages."""
    dev = torch.device("cuda", 0)
    B, Hq, Hkv, d = 64, 32, 8, 128
    max_pages = (1 << 31) // (Hkv * P * d * B) + 1
    num_pages = B * max_pages
    g = torch.Generator(device=dev).manual_seed(P)
    q = torch.empty(B, Hq, d, dtype=torch.bfloat16, device=dev).normal_(generator=g)
    kp = torch.empty(num_pages, Hkv, P, d, dtype=torch.bfloat16, device=dev).normal_(generator=g)
    vp = torch.empty(num_pages, Hkv, P, d, dtype=torch.bfloat16, device=dev).normal_(generator=g)
    table = torch.randperm(num_pages, generator=torch.Generator().manual_seed(P)).to(torch.int32)
    table = table.reshape(B, max_pages)
    lens = torch.full((B,), max_pages * P, dtype=torch.int32)
    lens[1] = 5
    o, lse = cuda_lib.decode_paged(q, kp, vp, table.to(dev), lens.to(dev), num_splits=0)
    torch.cuda.synchronize()
    st, detail = cuda_lib.fa_get_last_device_error()
    assert st == 0, detail
    for b in (0, 1, B - 1):
        n = int(lens[b])
        pages = table[b, :-(-n // P)].long()
        kb, vb = kp[pages.to(dev)].cpu(), vp[pages.to(dev)].cpu()
        tb = np.arange(pages.numel(), dtype=np.int32)[None]
        o_ref, lse_ref = naive.decode_paged(f64(q[b:b + 1].cpu()), f64(kb), f64(vb), tb,
                                            np.array([n], dtype=np.int32), 1 / math.sqrt(d))
        check_out(f64(o[b:b + 1].cpu()), f64(lse[b:b + 1].cpu()), o_ref, lse_ref, "P%d sequence %d" % (P, b))


@pytest.mark.parametrize("P,d", [(16, 128), (48, 128), (20, 128), (16, 64)])
def test_paged_decode_repeats_bits(cuda_lib, P, d):
    """B=32, Hq=32, Hkv=8, ragged lengths: 50 back-to-back calls give the first
    call's O and LSE bit for bit."""
    fa = cuda_lib
    dev = torch.device("cuda", 0)
    rng = np.random.default_rng(91 + P)
    lens = [4080, 1] + list(rng.integers(1, 4081, size=30))
    q, kp, vp, table, L = _case(92 + P + d, 32, 32, 8, P, lens, d)
    q, kp, vp = q.to(dev), kp.to(dev), vp.to(dev)
    table, L = torch.from_numpy(table).to(dev), torch.from_numpy(L).to(dev)
    o0, lse0 = fa.decode_paged(q, kp, vp, table, L)
    same = torch.ones((), dtype=torch.bool, device=dev)
    for _ in range(50):
        o, lse = fa.decode_paged(q, kp, vp, table, L)
        same &= (o.view(torch.int16) == o0.view(torch.int16)).all()
        same &= (lse.view(torch.int32) == lse0.view(torch.int32)).all()
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_error()[0] == 0
    assert bool(same)


@pytest.mark.parametrize("d", [128, 64])
def test_paged_decode_every_page_size_multiple_of_8(cuda_lib, d):
    """Every page size 8, 16, ..., 256 (boxes of gcd(page, 128) = 8 ... 128 rows on the
    tensor-core kernel), B=3, Hq=8, Hkv=2: a partial last page, a single token and a
    length past two 128-key stages, against the oracle."""
    for P in range(8, 264, 8):
        lens = [3 * P + 5, 1, 300]
        q, kp, vp, table, L = _case(500 + P + d, 3, 8, 2, P, lens, d)
        o, lse = _run(cuda_lib, q, kp, vp, table, L, 3)
        o_ref, lse_ref = naive.decode_paged(f64(q), f64(kp), f64(vp), table, L, 1 / math.sqrt(d))
        check_out(f64(o), f64(lse), o_ref, lse_ref, "page %d d%d" % (P, d))


@pytest.mark.parametrize("d", [128, 64])
def test_paged_decode_page_sizes_off_multiples_of_8(cuda_lib, d):
    """Page sizes that are not multiples of 8 (the CUDA-core kernel): 1 ... 7, odd,
    even, past a 128-key piece; B=3, Hq=8, Hkv=2, against the oracle."""
    for P in (1, 2, 3, 5, 7, 9, 12, 20, 33, 100, 130, 250):
        lens = [3 * P + 5, 1, 300]
        q, kp, vp, table, L = _case(700 + P + d, 3, 8, 2, P, lens, d)
        o, lse = _run(cuda_lib, q, kp, vp, table, L, 3)
        o_ref, lse_ref = naive.decode_paged(f64(q), f64(kp), f64(vp), table, L, 1 / math.sqrt(d))
        check_out(f64(o), f64(lse), o_ref, lse_ref, "page %d d%d" % (P, d))
