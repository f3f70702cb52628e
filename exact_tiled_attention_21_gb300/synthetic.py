"""Seeded synthetic inputs: the only module shared by the tests, the bench and
the oracle-side checks.  It draws numbers and describes workloads; it holds none
of the attention arithmetic.

Every tensor is drawn head by head on the host: for tensor ``tag`` and head
``(b, h)`` a ``torch.Generator('cpu')`` is seeded with a value derived from
``(seed, tag, b, h)``, a float32 N(0, 1) block is drawn, multiplied by ``std``
and rounded to bf16 (round-to-nearest-even, torch's conversion).  Any single
head can therefore be regenerated without drawing the others, which is how
the fp64 oracle gets bit-identical inputs for the heads it checks at full size.
"""
import math

import torch

TAG_Q, TAG_K, TAG_V, TAG_DO = 1, 2, 3, 4


def head_seed(seed, tag, b, h):
    """Seed of the generator stream for one (tensor, batch, head)."""
    return ((int(seed) * 131 + int(tag)) * 4099 + int(b)) * 4099 + int(h)


def head(seed, tag, b, h, n, d, std=1.0):
    """One head's [n, d] bf16 block (CPU)."""
    g = torch.Generator("cpu").manual_seed(head_seed(seed, tag, b, h))
    x = torch.randn((n, d), generator=g, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    return x.to(torch.bfloat16)


def bhnd(seed, tag, B, H, n, d, std=1.0):
    """A full [B, H, n, d] bf16 tensor (CPU), head by head."""
    out = torch.empty((B, H, n, d), dtype=torch.bfloat16)
    for b in range(B):
        for h in range(H):
            out[b, h] = head(seed, tag, b, h, n, d, std)
    return out


def bhd(seed, tag, B, H, d, std=1.0):
    """A [B, H, d] bf16 tensor (one row per head, e.g. a decode query)."""
    return bhnd(seed, tag, B, H, 1, d, std)[:, :, 0, :].contiguous()


def sample_rows(seed, n, count, must=(0,)):
    """``count`` distinct sorted row indices in [0, n), seeded, always holding
    ``must`` (clipped to range) and the last row n - 1."""
    g = torch.Generator("cpu").manual_seed(int(seed) * 7 + 11)
    keep = {min(max(int(m), 0), n - 1) for m in must} | {n - 1}
    perm = torch.randperm(n, generator=g).tolist()
    for r in perm:
        if len(keep) >= min(count, n):
            break
        keep.add(r)
    return sorted(keep)


def sample_heads(seed, H, count):
    """``count`` distinct head indices, seeded."""
    g = torch.Generator("cpu").manual_seed(int(seed) * 13 + 5)
    return sorted(torch.randperm(H, generator=g)[:count].tolist())


# The five workloads.  Shapes, distributions and seeds only.
CONFIGS = {
    "fwd_small": dict(kind="fwd", B=1, H=2, Nq=128, Nk=128, d=64, std=1.0, seed=0,
                      causal=(False,)),
    "fwd_4k": dict(kind="fwd", B=2, H=32, Nq=4096, Nk=4096, d=128, std=1.0, seed=1,
                   causal=(False, True)),
    "fwd_bwd_sweep": dict(kind="fwd_bwd", B=1, H=32, N=(1024, 2048, 4096, 8192), d=128,
                          std=1.0, seed=2, causal=(True,)),
    "decode": dict(kind="decode", B=32, H=32, Nk=4096, d=128, std=1.0, seed=3, splits=16),
    "long_causal": dict(kind="fwd", B=1, H=32, Nq=131072, Nk=131072, d=128, std=0.5, seed=4,
                        causal=(True,), sample_rows=64, sample_heads=4),
}


def head_f32(seed, tag, b, h, n, d, std=1.0):
    """One head's [n, d] float32 block (CPU), unrounded: the source of FP8 inputs."""
    g = torch.Generator("cpu").manual_seed(head_seed(seed, tag, b, h))
    x = torch.randn((n, d), generator=g, dtype=torch.float32)
    return x * std if std != 1.0 else x


def to_e4m3(x, rows=None):
    """Quantise float32 [B, H, N, d] to e4m3 bytes with fp32 scales.

    rows=None: one scale per head, shape [B*H]; otherwise one scale per
    ``rows``-row block of each head, shape [B*H, ceil(N/rows)].  A scale is the
    block's largest magnitude / 448 (1 for an all-zero block), and the stored
    byte is torch's round-to-nearest e4m3 of x / scale.  Returns
    (uint8 [B, H, N, d], float32 scales).  Input preparation only: the value an
    element stands for is e4m3(byte) * scale."""
    B, H, N, d = x.shape
    xs = x.reshape(B * H, N, d)
    if rows is None:
        amax = xs.abs().amax(dim=(1, 2))
        sc = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
        q = xs / sc[:, None, None]
    else:
        nb = -(-N // rows)
        pad = torch.zeros(B * H, nb * rows, d)
        pad[:, :N] = xs
        amax = pad.reshape(B * H, nb, rows, d).abs().amax(dim=(2, 3))
        sc = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
        q = (pad.reshape(B * H, nb, rows, d) / sc[:, :, None, None]).reshape(B * H, nb * rows, d)[:, :N]
    q = q.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    return q.reshape(B, H, N, d).contiguous(), sc.float().contiguous()


def default_scale(d):
    """The scale the workloads use: 1/sqrt(d)."""
    return 1.0 / math.sqrt(d)
