"""The C-ABI library: builds, loads, exports every declared symbol, and rejects
bad arguments before launching anything (these run without a GPU)."""
import ctypes

import pytest

import exact_tiled_attention_21_gb300 as fa


@pytest.fixture(scope="module")
def lib():
    fa.build()
    return fa.load()


def test_exports_every_declared_symbol(lib):
    names = fa.declared_symbols()
    assert {"fa_fwd", "fa_bwd", "fa_decode", "fa_bwd_workspace_bytes", "fa_decode_workspace_bytes",
            "fa_get_last_device_error", "fa_status_string", "fa_version",
            "fa_set_wait_timeout_ns"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for st in range(0, -7, -1):
        assert fa.fa_status_string(st)
    assert fa.fa_version() >= 100


def test_workspace_queries(lib):
    B, H, N, d = 2, 3, 1000, 128
    ws = fa.fa_bwd_workspace_bytes(B, H, N, N, d)
    assert ws >= B * H * N * 4
    assert fa.fa_bwd_workspace_bytes(B, H, N, N, 96) == 0
    assert fa.fa_bwd_workspace_bytes(0, H, N, N, d) == 0
    assert fa.fa_decode_workspace_bytes(32, 32, 4096, 128, 16) >= 32 * 32 * 16 * (128 + 1) * 4
    assert fa.fa_decode_workspace_bytes(1, 1, 1, 64, 0) > 0
    assert fa.fa_decode_workspace_bytes(1, 1, 10, 64, 300) == 0


def _fwd(lib, q=16, k=16, v=16, o=16, lse=16, B=1, H=1, Nq=8, Nk=8, d=64, scale=0.125, causal=0):
    return lib.fa_fwd(ctypes.c_void_p(q), ctypes.c_void_p(k), ctypes.c_void_p(v), ctypes.c_void_p(o),
                      ctypes.c_void_p(lse), B, H, Nq, Nk, d, scale, causal, None)


def test_forward_validation(lib):
    # every case is rejected on the host, before any CUDA call
    assert _fwd(lib, q=0) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, lse=0) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, Nq=0) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, B=-1) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, scale=float("nan")) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, scale=0.0) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, causal=2) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, d=96) == fa.FA_ERR_UNSUPPORTED
    assert _fwd(lib, d=256) == fa.FA_ERR_UNSUPPORTED
    assert _fwd(lib, k=24) == fa.FA_ERR_ALIGNMENT
    assert _fwd(lib, o=18) == fa.FA_ERR_ALIGNMENT


def test_backward_and_decode_validation(lib):
    vp = ctypes.c_void_p
    p = [vp(16)] * 9
    ws_need = fa.fa_bwd_workspace_bytes(1, 1, 8, 8, 64)
    assert lib.fa_bwd(*p, 1, 1, 8, 8, 64, 0.125, 0, vp(16), ws_need - 1, None) == fa.FA_ERR_WORKSPACE
    assert lib.fa_bwd(*p, 1, 1, 8, 8, 64, 0.125, 0, None, ws_need, None) == fa.FA_ERR_WORKSPACE
    assert lib.fa_bwd(*p, 1, 1, 8, 8, 64, 0.125, 0, vp(8), ws_need, None) == fa.FA_ERR_ALIGNMENT
    assert lib.fa_bwd(*([vp(0)] + p[1:]), 1, 1, 8, 8, 64, 0.125, 0, vp(16), ws_need, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_bwd(*p, 1, 1, 8, 8, 80, 0.125, 0, vp(16), ws_need, None) == fa.FA_ERR_UNSUPPORTED
    pr = [vp(16)] * 8
    assert lib.fa_bwd_dkdv_pair(*([vp(0)] + pr[1:]), 1, 1, 8, 8, 128, 0.125, 0, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_bwd_dkdv_pair(*pr, 1, 1, 8, 8, 64, 0.125, 0, None) == fa.FA_ERR_UNSUPPORTED  # pairs: d = 128
    assert lib.fa_bwd_dkdv_pair(*pr, 1, 1, 8, 8, 80, 0.125, 0, None) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_bwd_dkdv_pair(*pr, 1, 1, 8, 8, 128, 0.125, 2, None) == fa.FA_ERR_INVALID_ARG
    d_need = fa.fa_decode_workspace_bytes(2, 2, 100, 128, 16)
    q = [vp(16)] * 5
    assert lib.fa_decode(*q, 2, 2, 100, 128, 0.1, 16, vp(16), d_need - 4, None) == fa.FA_ERR_WORKSPACE
    assert lib.fa_decode(*q, 2, 2, 100, 128, 0.1, 300, vp(16), d_need, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_decode(*q, 2, 2, 0, 128, 0.1, 16, vp(16), d_need, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_decode(*q[:4], vp(20), 2, 2, 100, 128, 0.1, 16, vp(16), d_need, None) == fa.FA_ERR_ALIGNMENT


def test_selftest_argument_checks(lib):
    fn = lib.fa_selftest_wait_timeout
    fn.argtypes = [ctypes.c_uint64, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    assert fn(10, None) == fa.FA_ERR_INVALID_ARG              # below 1 us
    assert fn(5_000_000_000, None) == fa.FA_ERR_INVALID_ARG   # above 1 s


def test_wait_timeout_setting(lib):
    old = fa.fa_set_wait_timeout_ns(5_000_000)
    assert fa.fa_set_wait_timeout_ns(10) == 5_000_000    # raised to the 1 ms floor next
    assert fa.fa_set_wait_timeout_ns(old) == 1_000_000


def test_product_path_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(fa, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(fa, "_lib", None)
    with pytest.raises(fa.FAError):
        fa.load()


@pytest.mark.parametrize("per_chunk", [False, True])
def test_work_schedule_is_a_partition(lib, per_chunk):
    """Every work item of the persistent grids is taken by exactly one CTA, for
    chunks larger and smaller than the grid, ragged last chunks and rounds;
    without per-chunk rounds every CTA's count is within one item."""
    for n_items, chunk, grid in [(1, 1, 1), (5, 2, 3), (512, 512, 152), (2048, 1024, 152), (2048, 32, 152),
                                 (4096, 512, 152), (4097, 333, 152), (256, 8, 152), (100, 100, 152),
                                 (16384, 512, 152), (3, 64, 2)]:
        g = min(grid, n_items)
        owner = fa.fa_work_schedule(n_items, chunk, g, per_chunk)
        assert len(owner) == n_items and all(0 <= c < g for c in owner), (n_items, chunk, g)
        counts = [0] * g
        for c in owner:
            counts[c] += 1
        assert sum(counts) == n_items
        if not per_chunk or chunk < g:
            assert max(counts) - min(counts) <= 1, (n_items, chunk, g, max(counts), min(counts))


def test_work_schedule_balances_causal_chunks(lib):
    """Causal lists (each chunk heaviest first: 16 heads of 64 key tiles whose
    weights fall from 64 to 1): per-chunk rounds keep the busiest CTA within 2%
    of the mean, where rounds over the whole list would give it ~10% more."""
    heads, tiles, g = 16, 64, 152
    weights = [tiles - (i // heads) for i in range(heads * tiles)] * 2  # two chunks
    for per_chunk, bound in ((True, 1.02), (False, None)):
        owner = fa.fa_work_schedule(len(weights), heads * tiles, g, per_chunk)
        load = [0] * g
        for w, c in zip(weights, owner):
            load[c] += w
        ratio = max(load) / (sum(load) / g)
        if bound:
            assert ratio <= bound, ratio
        else:
            assert ratio > 1.05, ratio  # the reason for per-chunk rounds


def test_work_schedule_rejects_bad_sizes(lib):
    with pytest.raises(fa.FAError):
        fa.fa_work_schedule(10, 0, 4, True)
    with pytest.raises(fa.FAError):
        fa.fa_work_schedule(10, 4, 0, False)
