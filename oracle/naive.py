"""O1 — naive materialised attention in numpy fp64.  TEST INFRASTRUCTURE ONLY.

What is computed (the plain definition, applied to inputs widened exactly to fp64):

    S = scale * Q K^T                    [AIE "Das Grundproblem"; JOHE "Введение"]
    P = softmax(S) over the key axis     (masked entries contribute nothing)
    O = P V
    LSE_i = log sum_j exp(S_ij)          (natural log, over the allowed keys)

The pages write the transpose of K as ``K.T`` on 4-D tensors ([AIE]) and as
``K.transpose(-2, -3)`` in the "Проблема 1" listing of [JOHE]; both are read as
the transpose of the last two axes, which is what [JOHE]'s benchmark section
uses.  The causal mask ([ZIMA] "Kernel-Fusion ..." lists masking among the fused
steps) is aligned bottom-right: query i may see key j iff j <= i + (Nk - Nq).
For Nq == Nk this is the usual j <= i.  A query that sees no key at all
(only possible when causal and Nq > Nk) gets O = 0 and LSE = -inf.

Backward (gradient of the forward for an upstream dO; [JOHE] "Стадии
вычисления", pass 2 recomputes these from the same blocks without storing P —
here P is simply materialised):

    dV = P^T dO
    dP = dO V^T
    dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik)        (softmax Jacobian)
    dQ = scale * dS K
    dK = scale * dS^T Q

Decode is the forward with a single query against a KV cache, non-causal
([ZIMA] "Weniger IO bedeutet nicht, dass der KV-Cache entfällt": the cache
stays, attention streams it).  ``decode_split`` states the split-KV form: each
contiguous chunk of keys gives a partial (normalised partial output, partial
LSE) and the partials merge with the same max-shift rule as the online
recurrence of [AIE] "Lösung: Online Softmax".
"""
import numpy as np


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def allowed(Nq, Nk, causal, rows=None, window=0):
    """Boolean [len(rows), Nk]: which keys each query row may attend to.

    ``rows`` are query indices in [0, Nq) (default: all).  Causal alignment is
    bottom-right (key j visible to query i iff j <= i + Nk - Nq).  A sliding
    window of w >= 1 keys (causal only; the local attention with a fixed
    window that johe.ru "Flash Attention: ...", section "Альтернативы",
    describes) also hides the keys j <= i + Nk - Nq - w: each query sees at most
    the w keys ending at its diagonal.
    """
    rows = np.arange(Nq) if rows is None else np.asarray(rows)
    cols = np.arange(Nk)
    if not causal:
        return np.ones((rows.size, Nk), dtype=bool)
    hi = rows[:, None] + (Nk - Nq)
    ok = cols[None, :] <= hi
    if window:
        ok &= cols[None, :] > hi - window
    return ok


def forward(q, k, v, scale, causal=False, rows=None, Nq=None, return_p=False, window=0):
    """Materialised forward.

    q: [..., R, d] query rows (R = Nq, or the sampled rows when ``rows`` given)
    k: [..., Nk, d], v: [..., Nk, dv]
    rows: optional query indices of the R given rows (for the causal mask);
          Nq: total number of queries (needed with ``rows`` for the causal offset).
    Returns O [..., R, dv], LSE [..., R] (and P when return_p).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    R, Nk = q.shape[-2], k.shape[-2]
    if rows is None:
        Nq = R
    mask = allowed(Nq, Nk, causal, rows, window)
    s = scale * (q @ np.swapaxes(k, -1, -2))
    s = np.where(mask, s, -np.inf)
    m = s.max(axis=-1, keepdims=True)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m_safe)                      # exp(-inf) = 0 for masked keys
    l = e.sum(axis=-1, keepdims=True)
    has = l > 0
    p = np.where(has, e / np.where(has, l, 1.0), 0.0)
    o = p @ v
    lse = np.where(has, m_safe + np.log(np.where(has, l, 1.0)), -np.inf)[..., 0]
    if return_p:
        return o, lse, p
    return o, lse


def backward(q, k, v, do, scale, causal=False, rows=None, Nq=None, window=0):
    """Gradients (dQ, dK, dV) of O = softmax(scale Q K^T [masked]) V for upstream dO.

    With ``rows`` (query indices of the given q / dO rows, ``Nq`` the total query
    count) the result is the contribution of those query rows only: dQ of those
    rows, and their share of dK and dV (the full dK, dV are the sums of the
    shares over any partition of the queries).
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    _, _, p = forward(q, k, v, scale, causal, rows=rows, Nq=Nq, return_p=True, window=window)
    dv = np.swapaxes(p, -1, -2) @ do
    dp = do @ np.swapaxes(v, -1, -2)
    ds = p * (dp - (p * dp).sum(axis=-1, keepdims=True))
    dq = scale * (ds @ k)
    dk = scale * (np.swapaxes(ds, -1, -2) @ q)
    return dq, dk, dv


def forward_varlen(q, k, v, lens_q, lens_k, scale, causal=False):
    """A padded batch of sequences of different lengths ([ZIMA] "Kernel-Fusion
    ...": masking applied to the scores; here the mask is the sequence's own
    extent).  q [B,H,Nq,d], k/v [B,H,Nk,d]; sequence b is q[b,:, :lens_q[b]]
    against k/v[b,:, :lens_k[b]], with the bottom-right causal alignment of its
    own lengths.  Rows past lens_q[b] are padding: O = 0, LSE = -inf."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Nq, _ = q.shape
    O = np.zeros(q.shape[:-1] + (v.shape[-1],))
    L = np.full((B, H, Nq), -np.inf)
    for b in range(B):
        nq, nk = int(lens_q[b]), int(lens_k[b])
        if nq == 0:
            continue
        if nk == 0:  # no key at all: every row sees nothing
            continue
        o, lse = forward(q[b, :, :nq], k[b, :, :nk], v[b, :, :nk], scale, causal)
        O[b, :, :nq] = o
        L[b, :, :nq] = lse
    return O, L


def backward_varlen(q, k, v, do, lens_q, lens_k, scale, causal=False):
    """Gradients of ``forward_varlen``: each sequence's slice as in ``backward``;
    padding rows of dQ, dK and dV are zero."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(q.shape[0]):
        nq, nk = int(lens_q[b]), int(lens_k[b])
        if nq == 0 or nk == 0:
            continue
        g = backward(q[b, :, :nq], k[b, :, :nk], v[b, :, :nk], do[b, :, :nq], scale, causal)
        dq[b, :, :nq], dk[b, :, :nk], dv[b, :, :nk] = g
    return dq, dk, dv


def e4m3_value(byte):
    """The number an OCP e4m3 byte stands for (1 sign bit, 4 exponent bits with
    bias 7, 3 mantissa bits; exponent 0 is subnormal, 2^-6 * m/8; the pattern
    S.1111.111 is NaN; there are no infinities)."""
    b = int(byte)
    sign = -1.0 if b & 0x80 else 1.0
    e, m = (b >> 3) & 0xF, b & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


_E4M3 = np.array([e4m3_value(b) for b in range(256)])


def dequant_e4m3(x8, scales, rows=None):
    """fp64 values of e4m3 bytes [B,H,N,d] with one scale per head ([B*H]) or
    per ``rows``-row block of each head ([B*H, ceil(N/rows)])."""
    x8 = np.asarray(x8, dtype=np.uint8)
    B, H, N, d = x8.shape
    val = _E4M3[x8].reshape(B * H, N, d)
    sc = np.asarray(scales, dtype=np.float64)
    if rows is None:
        val = val * sc.reshape(B * H, 1, 1)
    else:
        val = val * np.repeat(sc.reshape(B * H, -1), rows, axis=1)[:, :N, None]
    return val.reshape(B, H, N, d)


def forward_fp8(q8, k8, v8, q_scale, k_scale, v_scale, scale, causal=False, rows=None, Nq=None):
    """The FP8 block-scaled forward ([JOHE] "Flash Attention 3": block-scaled
    attention; "Flash Attention 4": FP8) as the exact attention of the values
    the inputs stand for: q and k with one scale per 128-row block, v with one
    per head.  ``rows`` / ``Nq`` as in ``forward`` (q8 then holds those rows,
    and q_scale stays the full per-block array of the Nq rows)."""
    if rows is None:
        q = dequant_e4m3(q8, q_scale, rows=128)
    else:
        rows_a = np.asarray(rows)
        q8 = np.asarray(q8, dtype=np.uint8)
        B, H = q8.shape[:2]
        qsc = np.asarray(q_scale, dtype=np.float64).reshape(B * H, -1)[:, rows_a // 128]
        q = (_E4M3[q8].reshape(B * H, len(rows_a), -1) * qsc[:, :, None]).reshape(q8.shape)
    k = dequant_e4m3(k8, k_scale, rows=128)
    v = dequant_e4m3(v8, v_scale)
    return forward(q, k, v, scale, causal, rows=rows, Nq=Nq)


def decode(q, kcache, vcache, scale):
    """One query per (b, h) against its cache.  q [B,H,d], caches [B,H,Nk,d].

    Returns O [B,H,dv], LSE [B,H]: the forward with Nq = 1, non-causal.
    """
    o, lse = forward(_f64(q)[..., None, :], kcache, vcache, scale, causal=False)
    return o[..., 0, :], lse[..., 0]


def split_bounds(Nk, num_splits):
    """Contiguous key chunks [s*c, min((s+1)*c, Nk)) with c = ceil(Nk / num_splits).

    A chunk past the end is empty; its partial has LSE = -inf and weight 0.
    """
    c = -(-Nk // num_splits)
    return [(min(s * c, Nk), min((s + 1) * c, Nk)) for s in range(num_splits)]


def decode_split(q, kcache, vcache, scale, num_splits):
    """Split-KV decode written out: per-chunk partials, then the LSE merge.

    Partial of chunk s:  lse_s = log sum_{j in s} exp(x_j),  o_s = sum_j exp(x_j - lse_s) v_j
    Merge:               LSE = M + log sum_s exp(lse_s - M),  M = max_s lse_s
                         O   = sum_s exp(lse_s - LSE) o_s
    Returns (O, LSE, partial_o [B,H,S,dv], partial_lse [B,H,S]).
    """
    q, kc, vc = _f64(q), _f64(kcache), _f64(vcache)
    B, H, Nk, _ = kc.shape
    dv = vc.shape[-1]
    po = np.zeros((B, H, num_splits, dv))
    pl = np.full((B, H, num_splits), -np.inf)
    for s, (a, b) in enumerate(split_bounds(Nk, num_splits)):
        if b <= a:
            continue
        o, l = forward(q[..., None, :], kc[:, :, a:b], vc[:, :, a:b], scale)
        po[:, :, s] = o[..., 0, :]
        pl[:, :, s] = l[..., 0]
    m = pl.max(axis=-1, keepdims=True)
    w = np.exp(pl - m)
    lse = m[..., 0] + np.log(w.sum(axis=-1))
    o = (np.exp(pl - lse[..., None])[..., None] * po).sum(axis=-2)
    return o, lse, po, pl


def gather_pages(pages, block_table_row, length):
    """The first ``length`` tokens of one sequence from a paged cache.

    pages: [num_pages, page_size, dv] (one kv head); block_table_row: physical
    page of each logical page of the sequence, in order.
    """
    P = pages.shape[1]
    n = -(-length // P)
    rows = np.concatenate([pages[int(block_table_row[p])] for p in range(n)], axis=0) if n else pages[:0, 0]
    return rows[:length]


def decode_paged(q, k_pages, v_pages, block_table, seq_lens, scale):
    """Decode against a paged KV cache with grouped-query heads.

    q [B, Hq, d]; k_pages / v_pages [num_pages, Hkv, page_size, d];
    block_table [B, max_pages] (physical page of each logical page);
    seq_lens [B] (tokens in each sequence, >= 1).  Query head h reads kv head
    h // (Hq // Hkv).  Each (b, h) is the plain decode of its query against the
    sequence's tokens gathered in logical order (the cache is paged storage,
    not a different computation: PagedAttention in johe.ru "Flash Attention:
    ...", section "Альтернативы").  Returns O [B, Hq, dv], LSE [B, Hq].
    """
    q, kp, vp = _f64(q), _f64(k_pages), _f64(v_pages)
    B, Hq, _ = q.shape
    Hkv = kp.shape[1]
    g = Hq // Hkv
    o = np.zeros((B, Hq, vp.shape[-1]))
    lse = np.zeros((B, Hq))
    for b in range(B):
        L = int(seq_lens[b])
        for kvh in range(Hkv):
            K = gather_pages(kp[:, kvh], block_table[b], L)
            V = gather_pages(vp[:, kvh], block_table[b], L)
            oo, ll = forward(q[b, kvh * g:(kvh + 1) * g], K, V, scale)
            o[b, kvh * g:(kvh + 1) * g] = oo
            lse[b, kvh * g:(kvh + 1) * g] = ll
    return o, lse
