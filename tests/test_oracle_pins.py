"""Pins of the fp64 oracle against facts fixed by the pages and by mathematics.

Nothing here compares the oracle with itself: each check is a closed form, an
invariant, a library routine (torch SDPA / autograd in fp64), finite
differences, brute force on tiny inputs, or a hand-derived golden value under
tests/golden/.  ``test_planted_mistakes_are_caught`` plants plausible mistakes
in copies of the oracle and shows that some pin fails for each of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import naive, online, twopass

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")
RNG = np.random.default_rng(1234)


def _num(x):
    if isinstance(x, str):
        return {"ln3": math.log(3.0), "ln4": math.log(4.0), "-inf": -math.inf,
                "0.75ln3": 0.75 * math.log(3.0)}[x]
    return float(x)


def _arr(rows):
    return np.array([[_num(x) for x in r] for r in rows], dtype=np.float64)


def _fwd_impls():
    return {
        "naive": lambda q, k, v, s, c: naive.forward(q, k, v, s, c),
        "online": lambda q, k, v, s, c: tuple(np.array(x) for x in online.forward(q, k, v, s, c)),
        "twopass": lambda q, k, v, s, c: twopass.forward(q, k, v, s, c, block=3, nthreads=2),
    }


# ---------------------------------------------------------------- checkers
def check_golden_forward(fwd):
    cases = json.load(open(GOLDEN))["cases"]
    for c in cases:
        if "O" not in c:
            continue
        q, k, v = _arr(c["q"]), _arr(c["k"]), _arr(c["v"])
        o, lse = fwd(q, k, v, c["scale"], c["causal"])
        np.testing.assert_allclose(o, _arr(c["O"]), rtol=0, atol=1e-13, err_msg=c["name"])
        want = np.array([_num(x) for x in c["LSE"]])
        assert np.array_equal(np.isinf(lse), np.isinf(want)), c["name"]
        fin = np.isfinite(want)
        np.testing.assert_allclose(lse[fin], want[fin], rtol=0, atol=1e-13, err_msg=c["name"])


def check_golden_backward(bwd):
    c = [c for c in json.load(open(GOLDEN))["cases"] if c["name"] == "two_keys_backward"][0]
    dq, dk, dv = bwd(_arr(c["q"]), _arr(c["k"]), _arr(c["v"]), _arr(c["dO"]), c["scale"], c["causal"])
    np.testing.assert_allclose(dq, _arr(c["dQ"]), atol=1e-13, rtol=0)
    np.testing.assert_allclose(dk, _arr(c["dK"]), atol=1e-13, rtol=0)
    np.testing.assert_allclose(dv, _arr(c["dV"]), atol=1e-13, rtol=0)


def check_rows_sum_to_one(fwd_p):
    for Nq, Nk, causal in [(5, 9, False), (9, 5, False), (7, 7, True), (4, 11, True)]:
        q, k, v = RNG.standard_normal((2, Nq, 3)), RNG.standard_normal((2, Nk, 3)), RNG.standard_normal((2, Nk, 2))
        _, _, p = fwd_p(q, k, v, 0.7, causal)
        assert p.shape == (2, Nq, Nk)
        np.testing.assert_allclose(p.sum(-1), 1.0, atol=1e-12)
        assert (p >= 0).all()


def check_q_zero(fwd):
    Nk, d = 13, 4
    k, v = RNG.standard_normal((Nk, d)), RNG.standard_normal((Nk, 3))
    q = np.zeros((Nk, d))
    o, lse = fwd(q, k, v, 0.5, False)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(0), o.shape), atol=1e-12)
    np.testing.assert_allclose(lse, math.log(Nk), atol=1e-12)
    o, lse = fwd(q, k, v, 0.5, True)
    want = np.cumsum(v, 0) / np.arange(1, Nk + 1)[:, None]
    np.testing.assert_allclose(o, want, atol=1e-12)
    np.testing.assert_allclose(lse, np.log(np.arange(1, Nk + 1)), atol=1e-12)


def check_identical_keys(fwd):
    Nq, Nk, d = 6, 10, 5
    q = RNG.standard_normal((Nq, d))
    k = np.tile(RNG.standard_normal((1, d)), (Nk, 1))
    v = RNG.standard_normal((Nk, 4))
    o, lse = fwd(q, k, v, 0.3, False)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(0), o.shape), atol=1e-12)
    np.testing.assert_allclose(lse, math.log(Nk) + 0.3 * (q @ k[0]), atol=1e-12)


def check_single_key(fwd):
    q, k, v = RNG.standard_normal((4, 6)), RNG.standard_normal((1, 6)), RNG.standard_normal((1, 6))
    o, lse = fwd(q, k, v, 0.25, False)
    np.testing.assert_allclose(o, np.broadcast_to(v[0], o.shape), atol=1e-12)
    np.testing.assert_allclose(lse, 0.25 * (q @ k[0]), atol=1e-12)


def check_causal_first_row(fwd):
    N = 9
    q, k, v = RNG.standard_normal((N, 4)), RNG.standard_normal((N, 4)), RNG.standard_normal((N, 4))
    o, lse = fwd(q, k, v, 0.5, True)
    np.testing.assert_allclose(o[0], v[0], atol=1e-12)
    np.testing.assert_allclose(lse[0], 0.5 * q[0] @ k[0], atol=1e-12)
    # the last row of a square causal problem sees every key: equals non-causal
    o2, lse2 = fwd(q, k, v, 0.5, False)
    np.testing.assert_allclose(o[-1], o2[-1], atol=1e-12)
    np.testing.assert_allclose(lse[-1], lse2[-1], atol=1e-12)


def check_constant_v(fwd):
    q, k = RNG.standard_normal((5, 3)), RNG.standard_normal((8, 3))
    row = RNG.standard_normal(4)
    v = np.tile(row, (8, 1))
    for causal in (False, True):
        o, _ = fwd(q, k, v, 1.1, causal)
        np.testing.assert_allclose(o, np.broadcast_to(row, o.shape), atol=1e-12)


def check_key_shift(fwd):
    q, k, v = RNG.standard_normal((7, 4)), RNG.standard_normal((9, 4)), RNG.standard_normal((9, 3))
    u = RNG.standard_normal(4)
    for causal in (False, True):
        o, lse = fwd(q, k, v, 0.6, causal)
        o2, lse2 = fwd(q, k + u, v, 0.6, causal)
        np.testing.assert_allclose(o2, o, atol=1e-12)
        np.testing.assert_allclose(lse2, lse + 0.6 * (q @ u), atol=1e-12)


def check_permutation(fwd):
    q, k, v = RNG.standard_normal((6, 4)), RNG.standard_normal((11, 4)), RNG.standard_normal((11, 3))
    perm = RNG.permutation(11)
    o, lse = fwd(q, k, v, 0.4, False)
    o2, lse2 = fwd(q, k[perm], v[perm], 0.4, False)
    np.testing.assert_allclose(o2, o, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, atol=1e-12)


def check_finite_differences(bwd, fwd):
    """Central differences of L = sum(dO * O) at tiny sizes, relative error <= 1e-6."""
    h = 1e-6
    for Nq, Nk, d, causal in [(3, 4, 2, False), (4, 4, 3, True), (5, 3, 2, True), (2, 6, 4, True)]:
        q, k, v = RNG.standard_normal((Nq, d)), RNG.standard_normal((Nk, d)), RNG.standard_normal((Nk, d))
        do = RNG.standard_normal((Nq, d))
        scale = 0.8
        grads = bwd(q, k, v, do, scale, causal)

        def L(qq, kk, vv):
            return float((fwd(qq, kk, vv, scale, causal)[0] * do).sum())

        for which, g in zip(range(3), grads):
            args = [q, k, v]
            num = np.zeros_like(args[which])
            for idx in np.ndindex(*num.shape):
                plus = [a.copy() for a in args]
                minus = [a.copy() for a in args]
                plus[which][idx] += h
                minus[which][idx] -= h
                num[idx] = (L(*plus) - L(*minus)) / (2 * h)
            err = np.abs(num - g).max() / max(np.abs(num).max(), 1e-3)
            assert err <= 1e-6, (Nq, Nk, d, causal, which, err)


# ---------------------------------------------------------------- tests
@pytest.mark.parametrize("impl", ["naive", "online", "twopass"])
def test_golden_forward(impl):
    check_golden_forward(_fwd_impls()[impl])


def test_golden_backward():
    check_golden_backward(naive.backward)


def test_rows_sum_to_one():
    check_rows_sum_to_one(lambda q, k, v, s, c: naive.forward(q, k, v, s, c, return_p=True))


@pytest.mark.parametrize("impl", ["naive", "online", "twopass"])
@pytest.mark.parametrize("check", [check_q_zero, check_identical_keys, check_single_key,
                                   check_causal_first_row, check_constant_v, check_key_shift,
                                   check_permutation])
def test_closed_forms_and_invariants(impl, check):
    check(_fwd_impls()[impl])


@pytest.mark.parametrize("d", [4, 64])
@pytest.mark.parametrize("Nq,Nk", [(1, 1), (5, 5), (17, 17), (37, 37), (13, 29), (29, 13), (1, 37)])
@pytest.mark.parametrize("causal", [False, True])
def test_three_oracles_agree(d, Nq, Nk, causal):
    """O1 (materialised) = O2 (C two-pass) = O3 (online recurrence), 1e-12."""
    q, k, v = RNG.standard_normal((1, 2, Nq, d)), RNG.standard_normal((1, 2, Nk, d)), RNG.standard_normal((1, 2, Nk, d))
    scale = 1 / math.sqrt(d)
    o1, l1 = naive.forward(q, k, v, scale, causal)
    o2, l2 = twopass.forward(q, k, v, scale, causal, block=5, nthreads=3)
    for h in range(2):
        o3, l3 = online.forward(q[0, h], k[0, h], v[0, h], scale, causal, block=4)
        o3, l3 = np.array(o3), np.array(l3)
        np.testing.assert_allclose(o3, o1[0, h], atol=1e-12)
        fin = np.isfinite(l1[0, h])
        assert np.array_equal(fin, np.isfinite(l3))
        np.testing.assert_allclose(l3[fin], l1[0, h][fin], atol=1e-12)
    np.testing.assert_allclose(o2, o1, atol=1e-12)
    fin = np.isfinite(l1)
    assert np.array_equal(fin, np.isfinite(l2))
    np.testing.assert_allclose(l2[fin], l1[fin], atol=1e-12)


@pytest.mark.parametrize("Nq,Nk,causal", [(8, 8, False), (8, 8, True), (5, 12, True), (12, 5, False)])
def test_against_torch_sdpa_fp64(Nq, Nk, causal):
    """A library routine: torch's SDPA (math path, fp64 CPU) with an explicit mask."""
    q, k, v = RNG.standard_normal((2, 3, Nq, 8)), RNG.standard_normal((2, 3, Nk, 8)), RNG.standard_normal((2, 3, Nk, 8))
    scale = 0.35
    o, lse = naive.forward(q, k, v, scale, causal)
    mask = torch.ones(Nq, Nk, dtype=torch.bool)
    if causal:  # bottom-right alignment written independently with torch.tril's diagonal
        mask = torch.tril(mask, diagonal=Nk - Nq)
    tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=scale)
    np.testing.assert_allclose(o, ref.numpy(), atol=1e-12)
    s = (tq @ tk.transpose(-1, -2)) * scale
    ref_lse = torch.logsumexp(s.masked_fill(~mask, -math.inf), dim=-1)
    np.testing.assert_allclose(lse, ref_lse.numpy(), atol=1e-12)


def test_finite_differences():
    check_finite_differences(naive.backward, naive.forward)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_against_autograd_fp64(causal):
    """A library routine: torch autograd through fp64 SDPA."""
    Nq, Nk = 7, 10
    q, k, v, do = (RNG.standard_normal(s) for s in [(2, Nq, 8), (2, Nk, 8), (2, Nk, 8), (2, Nq, 8)])
    scale = 0.4
    dq, dk, dv = naive.backward(q, k, v, do, scale, causal)
    tq, tk, tv = (torch.from_numpy(x).requires_grad_() for x in (q, k, v))
    mask = torch.tril(torch.ones(Nq, Nk, dtype=torch.bool), diagonal=Nk - Nq) if causal else None
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=scale)
    out.backward(torch.from_numpy(do))
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_sums(causal):
    """sum_j dS_ij = 0 gives sum_j dK_j = 0; and sum_j dV_j = sum_i dO_i (every row sees a key)."""
    q, k, v, do = (RNG.standard_normal((3, 9, 5)) for _ in range(4))
    dq, dk, dv = naive.backward(q, k, v, do, 0.9, causal)
    np.testing.assert_allclose(dk.sum(-2), 0.0, atol=1e-12)
    np.testing.assert_allclose(dv.sum(-2), do.sum(-2), atol=1e-12)


def test_decode_is_last_row_of_forward():
    B, H, Nk, d = 2, 3, 21, 8
    kc, vc = RNG.standard_normal((B, H, Nk, d)), RNG.standard_normal((B, H, Nk, d))
    qs = RNG.standard_normal((B, H, Nk, d))
    o_full, lse_full = naive.forward(qs, kc, vc, 0.3, causal=True)  # last query sees the whole cache
    o, lse = naive.decode(qs[:, :, -1], kc, vc, 0.3)
    np.testing.assert_allclose(o, o_full[:, :, -1], atol=1e-12)
    np.testing.assert_allclose(lse, lse_full[:, :, -1], atol=1e-12)


@pytest.mark.parametrize("Nk,splits", [(64, 16), (37, 16), (5, 16), (1, 4), (100, 7), (4096, 16)])
def test_decode_split_equals_unsplit(Nk, splits):
    B, H, d = 2, 2, 8
    q = RNG.standard_normal((B, H, d))
    kc, vc = RNG.standard_normal((B, H, Nk, d)), RNG.standard_normal((B, H, Nk, d))
    o, lse = naive.decode(q, kc, vc, 0.5)
    o2, lse2, po, pl = naive.decode_split(q, kc, vc, 0.5, splits)
    np.testing.assert_allclose(o2, o, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, atol=1e-12)
    bounds = naive.split_bounds(Nk, splits)
    covered = [j for a, b in bounds for j in range(a, b)]
    assert covered == list(range(Nk))                 # disjoint, ordered, complete
    for s, (a, b) in enumerate(bounds):
        assert np.isinf(pl[..., s]).all() == (b <= a)  # empty chunk <=> lse = -inf


def test_sampled_rows_match_full():
    Nq = Nk = 40
    q, k, v = RNG.standard_normal((2, Nq, 8)), RNG.standard_normal((2, Nk, 8)), RNG.standard_normal((2, Nk, 8))
    rows = [0, 3, 17, 39]
    o, lse = naive.forward(q, k, v, 0.3, True)
    o1, l1 = naive.forward(q[:, rows], k, v, 0.3, True, rows=rows, Nq=Nq)
    o2, l2 = twopass.forward(q[:, rows], k, v, 0.3, True, rows=rows, Nq=Nq)
    for oo, ll in ((o1, l1), (o2, l2)):
        np.testing.assert_allclose(oo, o[:, rows], atol=1e-12)
        np.testing.assert_allclose(ll, lse[:, rows], atol=1e-12)


def test_backward_row_shares_add_up():
    """dK, dV are sums over queries: the shares of a partition of the query
    rows add up to the full gradient, and each share's dQ rows are the full dQ rows."""
    Nq, Nk = 23, 17
    q, k, v, do = (RNG.standard_normal(s) for s in [(2, Nq, 6), (2, Nk, 6), (2, Nk, 6), (2, Nq, 6)])
    for causal in (False, True):
        dq, dk, dv = naive.backward(q, k, v, do, 0.7, causal)
        sk, sv = np.zeros_like(dk), np.zeros_like(dv)
        for part in ([0, 5, 9], list(range(1, 5)), list(range(10, 23)), [6, 7, 8]):
            pq, pk, pv = naive.backward(q[:, part], k, v, do[:, part], 0.7, causal, rows=part, Nq=Nq)
            np.testing.assert_allclose(pq, dq[:, part], atol=1e-12)
            sk += pk
            sv += pv
        np.testing.assert_allclose(sk, dk, atol=1e-12)
        np.testing.assert_allclose(sv, dv, atol=1e-12)


def _paged_case(B, Hkv, g, P, lens, d, pages_extra=3, seed=7):
    rng = np.random.default_rng(seed)
    maxp = max(-(-L // P) for L in lens)
    npages = B * maxp + pages_extra
    kp, vp = rng.standard_normal((npages, Hkv, P, d)), rng.standard_normal((npages, Hkv, P, d))
    table = rng.permutation(npages)[:B * maxp].reshape(B, maxp)
    q = rng.standard_normal((B, Hkv * g, d))
    return q, kp, vp, table, np.array(lens)


def test_paged_decode_equals_contiguous_decode():
    """Identity page table, full lengths, one query head per kv head: the
    plain contiguous decode."""
    B, H, P, d, npg = 2, 3, 8, 16, 5
    q = RNG.standard_normal((B, H, d))
    kc, vc = RNG.standard_normal((B, H, P * npg, d)), RNG.standard_normal((B, H, P * npg, d))
    # pages [B*npg, H, P, d]: sequence b's logical page p is physical page b*npg + p
    kp = kc.reshape(B, H, npg, P, d).transpose(0, 2, 1, 3, 4).reshape(B * npg, H, P, d)
    vp = vc.reshape(B, H, npg, P, d).transpose(0, 2, 1, 3, 4).reshape(B * npg, H, P, d)
    table = np.arange(B * npg).reshape(B, npg)
    o, lse = naive.decode_paged(q, kp, vp, table, [P * npg] * B, 0.3)
    o2, lse2 = naive.decode(q, kc, vc, 0.3)
    np.testing.assert_allclose(o, o2, atol=1e-12)
    np.testing.assert_allclose(lse, lse2, atol=1e-12)


def test_paged_decode_invariances():
    """Moving pages to other physical slots (table updated) changes nothing;
    a sequence of length L equals decode against its first L tokens; the
    query heads of a group all read the same kv head."""
    q, kp, vp, table, lens = _paged_case(3, 2, 4, 8, [1, 13, 24], 16)
    o, lse = naive.decode_paged(q, kp, vp, table, lens, 0.25)
    perm = RNG.permutation(kp.shape[0])
    inv = np.argsort(perm)
    o2, lse2 = naive.decode_paged(q, kp[perm], vp[perm], inv[table], lens, 0.25)
    np.testing.assert_allclose(o2, o, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, atol=1e-12)
    for b in range(3):
        for h in range(8):
            K = np.concatenate([kp[table[b, p], h // 4] for p in range(table.shape[1])])[:lens[b]]
            V = np.concatenate([vp[table[b, p], h // 4] for p in range(table.shape[1])])[:lens[b]]
            oo, ll = naive.forward(q[b, h][None], K, V, 0.25)
            np.testing.assert_allclose(o[b, h], oo[0], atol=1e-12)
            np.testing.assert_allclose(lse[b, h], ll[0], atol=1e-12)
    # a single-token sequence returns that token's value, LSE = its score
    K0, V0 = kp[table[0, 0], 0, 0], vp[table[0, 0], 0, 0]
    np.testing.assert_allclose(o[0, 0], V0, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], 0.25 * q[0, 0] @ K0, atol=1e-12)


@pytest.mark.parametrize("Nq,Nk", [(9, 9), (5, 12), (12, 5)])
def test_sliding_window_pins(Nq, Nk):
    """A window of >= Nk keys is plain causal; a window of 1 key gives
    O_i = V[i + Nk - Nq] and LSE_i = its score; any window equals torch SDPA
    with the explicit band mask; rows sum to one over the band."""
    q, k, v = RNG.standard_normal((2, Nq, 6)), RNG.standard_normal((2, Nk, 6)), RNG.standard_normal((2, Nk, 5))
    off = Nk - Nq
    o_c, l_c = naive.forward(q, k, v, 0.4, True)
    o_w, l_w = naive.forward(q, k, v, 0.4, True, window=Nk + 3)
    np.testing.assert_allclose(o_w, o_c, atol=1e-12)
    np.testing.assert_allclose(l_w, l_c, atol=1e-12)
    o1, l1 = naive.forward(q, k, v, 0.4, True, window=1)
    for i in range(Nq):
        j = i + off
        if 0 <= j < Nk:
            np.testing.assert_allclose(o1[:, i], v[:, j], atol=1e-12)
            np.testing.assert_allclose(l1[:, i], 0.4 * (q[:, i] * k[:, j]).sum(-1), atol=1e-12)
        else:
            assert np.all(o1[:, i] == 0) and np.all(np.isneginf(l1[:, i]))
    for w in (2, 3, 5):
        o, lse, p = naive.forward(q, k, v, 0.4, True, window=w, return_p=True)
        band = torch.ones(Nq, Nk, dtype=torch.bool).tril(diagonal=off) & ~torch.ones(Nq, Nk, dtype=torch.bool).tril(diagonal=off - w)
        has = band.any(-1).numpy()
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[:, has]), torch.from_numpy(k), torch.from_numpy(v), attn_mask=band[has], scale=0.4)
        np.testing.assert_allclose(o[:, has], ref.numpy(), atol=1e-12)
        np.testing.assert_allclose(p[:, has].sum(-1), 1.0, atol=1e-12)
        assert (p[:, ~has] == 0).all()


def test_sliding_window_backward_finite_differences():
    def fwd_w(q, k, v, s, c):
        return naive.forward(q, k, v, s, c, window=3)
    def bwd_w(q, k, v, do, s, c):
        return naive.backward(q, k, v, do, s, c, window=3)
    check_finite_differences(bwd_w, fwd_w)


# ---------------------------------------------------------------- per-sequence lengths
VL_LENS = [(5, 7), (0, 4), (3, 0), (6, 2), (2, 9)]  # (len_q, len_k) per sequence; Nq = 6, Nk = 9


def _vl_case(causal_dim=6):
    B, H, Nq, Nk, d = len(VL_LENS), 2, 6, 9, causal_dim
    q, k = RNG.standard_normal((B, H, Nq, d)), RNG.standard_normal((B, H, Nk, d))
    v = RNG.standard_normal((B, H, Nk, 5))
    lq = np.array([a for a, _ in VL_LENS]); lk = np.array([b for _, b in VL_LENS])
    return q, k, v, lq, lk


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_closed_form_zero_query(causal):
    """Q = 0: row i < len_q sees keys [0, len_k) (causal: [0, i + len_k - len_q])
    with equal weights, so O_i is the mean of those V rows and LSE_i = ln(count);
    a row with no key, and every row past len_q, has O = 0 and LSE = -inf."""
    q, k, v, lq, lk = _vl_case()
    o, lse = naive.forward_varlen(np.zeros_like(q), k, v, lq, lk, 0.7, causal)
    for b, (nq, nk) in enumerate(VL_LENS):
        for i in range(q.shape[2]):
            cnt = 0 if i >= nq else (min(nk, i + nk - nq + 1) if causal else nk)
            cnt = max(cnt, 0)
            if cnt == 0:
                assert np.all(o[b, :, i] == 0) and np.all(np.isneginf(lse[b, :, i]))
            else:
                np.testing.assert_allclose(o[b, :, i], v[b, :, :cnt].mean(axis=1), atol=1e-12)
                np.testing.assert_allclose(lse[b, :, i], math.log(cnt), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_ignores_padding_and_matches_sdpa(causal):
    """Values in padding positions change nothing; each valid row equals torch
    SDPA with an explicit key-padding (and causal band) mask on the padded
    tensors."""
    q, k, v, lq, lk = _vl_case()
    o, lse = naive.forward_varlen(q, k, v, lq, lk, 0.7, causal)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    for b, (nq, nk) in enumerate(VL_LENS):
        q2[b, :, nq:] = 1e3
        k2[b, :, nk:] = -7.0
        v2[b, :, nk:] = 5e2
    o2, lse2 = naive.forward_varlen(q2, k2, v2, lq, lk, 0.7, causal)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)
    Nq, Nk = q.shape[2], k.shape[2]
    for b, (nq, nk) in enumerate(VL_LENS):
        i = torch.arange(Nq)[:, None]
        j = torch.arange(Nk)[None, :]
        mask = (j < nk) & (i < nq)
        if causal:
            mask &= j <= i + nk - nq
        has = mask.any(-1).numpy()
        if not has.any():
            continue
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q2[b][:, has]), torch.from_numpy(k2[b]), torch.from_numpy(v2[b]),
            attn_mask=mask[has], scale=0.7)
        np.testing.assert_allclose(o[b][:, has], ref.numpy(), atol=1e-12)


def test_varlen_full_lengths_equal_dense():
    q, k, v, _, _ = _vl_case()
    B, Nq, Nk = q.shape[0], q.shape[2], k.shape[2]
    for causal in (False, True):
        o, lse = naive.forward_varlen(q, k, v, [Nq] * B, [Nk] * B, 0.7, causal)
        o2, lse2 = naive.forward(q, k, v, 0.7, causal)
        np.testing.assert_allclose(o, o2, atol=1e-12)
        np.testing.assert_allclose(lse, lse2, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_backward_finite_differences(causal):
    """Central differences of L = sum(dO * O) through forward_varlen, over every
    input element including padding (whose gradient must be exactly zero)."""
    lens = [(3, 4), (2, 5), (0, 3)]
    B, H, Nq, Nk, d = len(lens), 1, 3, 5, 2
    q, k, v = RNG.standard_normal((B, H, Nq, d)), RNG.standard_normal((B, H, Nk, d)), RNG.standard_normal((B, H, Nk, d))
    do = RNG.standard_normal((B, H, Nq, d))
    lq = [a for a, _ in lens]; lk = [b for _, b in lens]
    grads = naive.backward_varlen(q, k, v, do, lq, lk, 0.8, causal)
    h = 1e-6

    def L(qq, kk, vv):
        o, _ = naive.forward_varlen(qq, kk, vv, lq, lk, 0.8, causal)
        return float((o * do).sum())

    for which, g in enumerate(grads):
        args = [q, k, v]
        num = np.zeros_like(args[which])
        for idx in np.ndindex(*num.shape):
            plus = [a.copy() for a in args]
            minus = [a.copy() for a in args]
            plus[which][idx] += h
            minus[which][idx] -= h
            num[idx] = (L(*plus) - L(*minus)) / (2 * h)
        assert np.abs(num - g).max() / max(np.abs(num).max(), 1e-3) <= 1e-6, (which, causal)
        for b, (nq, nk) in enumerate(lens):
            pad = g[b, :, (nq if which == 0 else nk):]
            assert np.all(pad == 0)


# ---------------------------------------------------------------- FP8 block-scaled forward
def test_e4m3_decoder_matches_library():
    """The oracle's decoder, written from the format (bias 7, 3 mantissa bits,
    subnormals, one NaN pattern per sign), equals torch's float8_e4m3fn for
    all 256 bytes."""
    lib = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([naive.e4m3_value(b) for b in range(256)])
    assert np.array_equal(np.isnan(lib), np.isnan(mine))
    assert np.array_equal(lib[~np.isnan(lib)], mine[~np.isnan(mine)])
    assert naive.e4m3_value(0x7E) == 448.0 and naive.e4m3_value(0x01) == 2.0 ** -9


def test_fp8_block_scales_and_folding():
    """Each 128-row block of q and k takes its own scale and v one per head:
    built element by element here; a factor moved from the q scales into the
    softmax scale changes nothing; sampled rows equal the full result."""
    from exact_tiled_attention_21_gb300 import synthetic as syn
    B, H, Nq, Nk, d = 1, 2, 200, 300, 8
    g = torch.Generator("cpu").manual_seed(5)
    q8, sq = syn.to_e4m3(torch.randn(B, H, Nq, d, generator=g) * 3, rows=128)
    k8, sk = syn.to_e4m3(torch.randn(B, H, Nk, d, generator=g), rows=128)
    v8, sv = syn.to_e4m3(torch.randn(B, H, Nk, d, generator=g))
    assert sq.shape == (B * H, 2) and sk.shape == (B * H, 3) and sv.shape == (B * H,)
    q = np.zeros((B, H, Nq, d)); k = np.zeros((B, H, Nk, d)); v = np.zeros((B, H, Nk, d))
    q8n, k8n, v8n = q8.numpy(), k8.numpy(), v8.numpy()
    for h in range(H):
        for i in range(Nq):
            q[0, h, i] = [naive.e4m3_value(x) * float(sq[h, i // 128]) for x in q8n[0, h, i]]
        for j in range(Nk):
            k[0, h, j] = [naive.e4m3_value(x) * float(sk[h, j // 128]) for x in k8n[0, h, j]]
            v[0, h, j] = [naive.e4m3_value(x) * float(sv[h]) for x in v8n[0, h, j]]
    for causal in (False, True):
        o8, l8 = naive.forward_fp8(q8n, k8n, v8n, sq.numpy(), sk.numpy(), sv.numpy(), 0.3, causal)
        o, l = naive.forward(q, k, v, 0.3, causal)
        np.testing.assert_allclose(o8, o, atol=1e-12)
        np.testing.assert_allclose(l8, l, atol=1e-12)
        o2, l2 = naive.forward_fp8(q8n, k8n, v8n, 2 * sq.numpy(), sk.numpy(), sv.numpy(), 0.15, causal)
        np.testing.assert_allclose(o2, o, atol=1e-12)
        np.testing.assert_allclose(l2, l, atol=1e-12)
        rows = [0, 127, 128, 199]
        o3, l3 = naive.forward_fp8(q8n[:, :, rows], k8n, v8n, sq.numpy(), sk.numpy(), sv.numpy(), 0.3, causal,
                                   rows=rows, Nq=Nq)
        np.testing.assert_allclose(o3, o[:, :, rows], atol=1e-12)
        np.testing.assert_allclose(l3, l[:, :, rows], atol=1e-12)


def test_e4m3_quantiser_error():
    """The input generator's quantiser: each value is within half an e4m3 step
    of x / scale (relative 2^-4, or 2^-10 absolute in the subnormal range)."""
    from exact_tiled_attention_21_gb300 import synthetic as syn
    x = torch.randn(1, 3, 300, 16, generator=torch.Generator("cpu").manual_seed(9)) * 5
    for rows in (None, 128):
        x8, sc = syn.to_e4m3(x, rows=rows)
        deq = naive.dequant_e4m3(x8.numpy(), sc.numpy(), rows=rows)
        xs = x.double().numpy()
        if rows is None:
            s_el = np.repeat(sc.double().numpy(), 300 * 16).reshape(1, 3, 300, 16)
        else:
            s_el = np.repeat(sc.double().numpy(), 128, axis=1)[:, :300].reshape(1, 3, 300, 1) * np.ones((1, 1, 1, 16))
        err = np.abs(deq - xs) / s_el
        assert np.all(err <= np.maximum(2.0 ** -4 * np.abs(xs) / s_el, 2.0 ** -10) + 1e-9)


# ---------------------------------------------------------------- mutation check
def _mutant_forward(kind):
    def fwd(q, k, v, scale, causal=False, return_p=False):
        q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
        Nq, Nk = q.shape[-2], k.shape[-2]
        mask = naive.allowed(Nq, Nk, causal)
        if kind == "top_left_causal" and causal:
            mask = np.tril(np.ones((Nq, Nk), dtype=bool))
        if kind == "reversed_causal" and causal:
            mask = mask[::-1, ::-1]
        sc = 1.0 if kind == "no_scale" else scale
        s = sc * (q @ np.swapaxes(k, -1, -2))
        s = np.where(mask, s, -np.inf)
        axis = -2 if kind == "softmax_wrong_axis" else -1
        m = s.max(axis=axis, keepdims=True)
        m = np.where(np.isfinite(m), m, 0.0)
        e = np.exp(s - m)
        l = e.sum(axis=axis, keepdims=True)
        p = np.where(l > 0, e / np.where(l > 0, l, 1), 0)
        if kind == "no_normalise":
            p = e
        o = p @ v
        # row statistics of the (possibly mutated) weights
        mr = np.where(np.isfinite(s.max(-1)), s.max(-1), 0.0)
        lr = np.exp(s - mr[..., None]).sum(-1)
        lse = np.where(lr > 0, mr + np.log(np.where(lr > 0, lr, 1)), -np.inf)
        if kind == "lse_log2":
            lse = lse / math.log(2)
        return (o, lse, p) if return_p else (o, lse)
    return fwd


def _mutant_backward(kind):
    def bwd(q, k, v, do, scale, causal=False):
        q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
        _, _, p = naive.forward(q, k, v, scale, causal, return_p=True)
        dv = np.swapaxes(p, -1, -2) @ do
        dp = do @ np.swapaxes(v, -1, -2)
        if kind == "no_rowsum_term":
            ds = p * dp
        elif kind == "wrong_sign":
            ds = p * (dp + (p * dp).sum(-1, keepdims=True))
        else:
            ds = p * (dp - (p * dp).sum(-1, keepdims=True))
        dq = scale * (ds @ k)
        dk = (np.swapaxes(ds, -1, -2) @ q) * (1.0 if kind == "dk_no_scale" else scale)
        if kind == "dv_transposed_p":
            dv = p[..., : dv.shape[-2], :] @ do if p.shape[-1] == p.shape[-2] else dv * 0
        return dq, dk, dv
    return bwd


@pytest.mark.parametrize("kind", ["top_left_causal", "reversed_causal", "no_scale",
                                  "softmax_wrong_axis", "no_normalise", "lse_log2"])
def test_planted_forward_mistakes_are_caught(kind):
    fwd = _mutant_forward(kind)
    checks = [check_golden_forward, check_q_zero, check_single_key, check_causal_first_row,
              check_key_shift, check_constant_v,
              lambda f: check_rows_sum_to_one(lambda q, k, v, s, c: f(q, k, v, s, c, return_p=True))]
    caught = 0
    for chk in checks:
        try:
            chk(fwd)
        except (AssertionError, ValueError):
            caught += 1
    assert caught > 0, kind


@pytest.mark.parametrize("kind", ["no_rowsum_term", "wrong_sign", "dk_no_scale", "dv_transposed_p"])
def test_planted_backward_mistakes_are_caught(kind):
    bwd = _mutant_backward(kind)
    with pytest.raises(AssertionError):
        check_finite_differences(bwd, naive.forward)
