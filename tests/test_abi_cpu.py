"""The C ABI on the CPU machine: the library loads, exports every declared symbol,
and its host-side contract agrees bit for bit with the oracle.  Refusals that
happen before any device work are checked here too (no GPU is touched: every
call below returns before the first CUDA call)."""
import ctypes
import os
import re

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from conftest import build_lib
    build_lib()
    import output_projection_cross_gb300 as L
    return L


def _declared():
    src = open(os.path.join(ROOT, "include", "lossk.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(lossk_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert len(names) >= 14
    lib = ctypes.CDLL(L.lossk.lib._name)
    for nm in names:
        assert hasattr(lib, nm), nm
    assert set(names) == set(L.lossk.EXPORTED)


def test_status_names_match_oracle(L):
    for code in range(570, 612):
        o = oracle.status_name(code)
        g = L.lossk_status_name(code)
        if code in (589, 590, 591, 592):
            assert o == "unknown_status"
            assert g in ("device_error", "device_timeout", "unaligned", "unknown_flags")
        else:
            assert g == o, code


@pytest.mark.parametrize("n,d,V", [(2048, 4096, 151936), (0, 4, 4), (1 << 16, 1 << 15, 1 << 15),
                                   ((1 << 16) + 1, 1 << 15, 1 << 15), ((1 << 24) + 1, 1, 1),
                                   (1, 1, 1), (5, -1, 3), (1 << 24, 1 << 22, 1)])
def test_dims_check_matches_oracle(L, n, d, V):
    assert L.lossk_dims_check(n, d, V) == oracle.dims_check(n, d, V)
    for ceiling in (0, 1, 1 << 46, (1 << 63) - 1):
        assert L.lossk_work_fits(n, d, V, ceiling) == oracle.work_fits(n, d, V, ceiling)


@pytest.mark.parametrize("chunk,V", [(256, 151936), (2048, 151936), (1 << 10, 1 << 17),
                                     ((1 << 10) + 1, 1 << 17), (0, 5), (5, 0), (1, 1 << 27),
                                     (2, 1 << 27), (883, 151936), (884, 151936)])
def test_chunk_check_matches_oracle(L, chunk, V):
    assert L.lossk_chunk_check(chunk, V) == oracle.chunk_check(chunk, V)
    assert L.lossk_logit_cells(chunk, V) == oracle.logit_cells(chunk, V)


@pytest.mark.parametrize("n,V,chunk", [(2048, 151936, 256), (100, 151936, 2048), (1000, 10, 3),
                                       (0, 10, 3), (7, 7, 7), (4096, 151936, 512)])
def test_peak_logit_cells_matches_oracle(L, n, V, chunk):
    assert L.lossk_peak_logit_cells(n, V, chunk) == oracle.peak_logit_cells(n, V, chunk)


def test_workspace_bytes(L):
    for kind in range(5):
        for dt in (0, 1):
            nb = L.lossk_workspace_bytes(kind, 2048, 1024, 151936, dt)
            assert nb > 0 and nb % 256 == 0
    assert L.lossk_workspace_bytes(0, 0, 1024, 151936, 1) == -1


def test_refusals_before_device_work(L):
    lib = L.lib
    P = 4096  # a 16-byte-aligned fake address: never dereferenced on these paths
    args = dict(n=64, d=64, V=1000)

    def fwd(n=64, d=64, V=1000, chunk=16, dtype=1, H=P, hl=64 * 64, W=P, wl=1000 * 64, y=P,
            yl=64, wz=0.0, lse=P, scal=P, ws=P, wsb=1 << 30):
        return lib.lossk_ce_fwd(n, d, V, chunk, dtype, H, hl, W, wl, y, yl, None, wz, lse, None,
                                scal, ws, wsb, None)

    assert fwd(n=0) == 581
    assert fwd(V=(1 << 24) + 1) == 583
    assert fwd(n=1 << 16, d=1 << 15, V=(1 << 15) + 8, hl=1 << 40, wl=1 << 40) == 584
    assert fwd(chunk=(1 << 27) // 1000 + 1) == 587
    assert fwd(chunk=0) == 581
    assert fwd(H=None) == 582
    assert fwd(hl=64 * 64 - 1) == 582
    assert fwd(yl=63) == 582
    assert fwd(wsb=255) == 582
    assert fwd(dtype=7) == 582
    assert fwd(H=P + 8) == 591
    assert fwd(d=60, hl=64 * 60, wl=1000 * 60) == 591      # bf16 rows need 16-byte pitch
    for wz in (float("nan"), float("inf"), -1.0):
        assert fwd(wz=wz) == 585
    # distillation: temperature and objective
    def dist(direction=0, T=1.0, wz=0.0, gs=1.0, Vv=1000, tl=64 * 1000):
        return lib.lossk_distill_fwd_bwd(64, 64, Vv, 16, 1, P, 64 * 64, P, Vv * 64, P, tl, None,
                                         direction, T, wz, gs, P, None, None, None, None, P,
                                         1 << 30, None)
    assert dist(T=0.0) == 585 and dist(T=-2.0) == 585 and dist(T=float("nan")) == 585
    assert dist(gs=float("inf")) == 585
    assert dist(direction=3) == 588 and dist(direction=-1) == 588
    assert dist(tl=10) == 582
    assert dist(Vv=1001, tl=64 * 1001) == 591   # bf16 teacher rows need 16-byte pitch
    # from logits
    assert lib.lossk_ce_from_logits(0, 10, 1, P, 0, P, 0, None, 0.0, 1.0, P, None, P, None, 0, P,
                                    1 << 20, None) == 581
    assert lib.lossk_ce_from_logits(4, 10, 1, P, 39, P, 4, None, 0.0, 1.0, P, None, P, None, 0, P,
                                    1 << 20, None) == 582
    out = L.lossk.lossk_peak_cells()
    assert lib.lossk_peak_logit_cells(1, 1, 1, None) == 582
