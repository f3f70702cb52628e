"""O3 — the online-softmax recurrence as a pure-Python loop.  TEST INFRASTRUCTURE ONLY.

Follows [AIE] "Lösung: Online Softmax" (wiki.ai-engineering.at, "Flash
Attention"), block by block over the keys, in fp64, for one query row at a time:

    m = -inf, l = 0, o = 0
    for each key block:
        S     = scores of the row against the block
        m_new = max(m, max(S))
        l     = exp(m - m_new) * l + sum(exp(S - m_new))
        o     = o * exp(m - m_new) + exp(S - m_new) @ V_block
        m     = m_new

The page stops there; the output is o / l after the last block (the reading
taken for the missing normalisation), and LSE = m + log(l).  The per-block
``softmax(S_ij)`` of the page's "Tiling Algorithm" listing is superseded by this
recurrence on the same page and is not used.  exp(-inf - (-inf)) is read as a
factor of 1 on an empty accumulator (nothing to rescale); a masked score is
-inf and contributes exp(-inf) = 0.  Only for small inputs (pure Python).
"""
import math


def _row(qrow, K, V, scale, allowed_cols, block):
    d = len(qrow)
    dv = len(V[0]) if V else 0
    m = -math.inf
    l = 0.0
    o = [0.0] * dv
    Nk = len(K)
    for j0 in range(0, Nk, block):
        cols = [j for j in range(j0, min(j0 + block, Nk)) if allowed_cols(j)]
        S = [scale * sum(qrow[c] * K[j][c] for c in range(d)) for j in cols]
        if not S:
            continue
        m_new = max(m, max(S))
        corr = 0.0 if m == -math.inf else math.exp(m - m_new)
        e = [math.exp(s - m_new) for s in S]
        l = corr * l + sum(e)
        o = [o[c] * corr + sum(e[t] * V[cols[t]][c] for t in range(len(cols)))
             for c in range(dv)]
        m = m_new
    if l == 0.0:
        return [0.0] * dv, -math.inf
    return [x / l for x in o], m + math.log(l)


def forward(q, k, v, scale, causal=False, block=4):
    """q [Nq][d], k [Nk][d], v [Nk][dv] nested lists (or arrays) for one head.

    Returns (O as list of rows, LSE list).  Causal alignment is bottom-right:
    key j visible to query i iff j <= i + Nk - Nq.
    """
    q = [list(map(float, r)) for r in q]
    k = [list(map(float, r)) for r in k]
    v = [list(map(float, r)) for r in v]
    Nq, Nk = len(q), len(k)
    O, L = [], []
    for i in range(Nq):
        lim = i + Nk - Nq
        ok = (lambda j, lim=lim: j <= lim) if causal else (lambda j: True)
        o, lse = _row(q[i], k, v, scale, ok, block)
        O.append(o)
        L.append(lse)
    return O, L
