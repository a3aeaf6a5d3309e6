"""lossk_ce_from_logits_static: the entry point for callers that cannot allocate.

Some callers (a plug-in whose device memory all belongs to its host framework's
arena, a runtime with a memory plan fixed at start-up) can neither allocate
nor hand the library a workspace.  This entry point keeps its scratch in a
device array built into the library.  The test calls it through the C ABI
twice in a row, on different inputs, and checks each result against the
workspace-based lossk_ce_from_logits within the tolerances the other tests
use (and, the kernels being the same, for identical bits).  It runs last so
that a failure here leaves every other test already run; it must pass both in
a fresh process and after the rest of the suite.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

BF16_LOSS, BF16_GRAD = 2e-3, 1e-2
F32_LOSS, F32_GRAD = 1e-6, 1e-5


@pytest.fixture(scope="module")
def L():
    from conftest import build_lib
    build_lib()
    import output_projection_cross_gb300 as L
    assert torch.cuda.is_available()
    return L


def _call_static(L, X, y, mask, wz, gs):
    """Through the C ABI directly: every output allocated here, before the call."""
    n, V = X.shape
    lse = torch.empty(n, dtype=torch.float32, device="cuda")
    ce = torch.empty(n, dtype=torch.float32, device="cuda")
    sc = torch.empty(3, dtype=torch.float64, device="cuda")
    g = torch.empty_like(X)
    dt = 1 if X.dtype == torch.bfloat16 else 0
    st = L.lib.lossk_ce_from_logits_static(
        n, V, dt, X.data_ptr(), X.numel(), y.data_ptr(), y.numel(),
        None if mask is None else mask.data_ptr(), wz, gs, lse.data_ptr(), ce.data_ptr(),
        sc.data_ptr(), g.data_ptr(), g.numel(), torch.cuda.current_stream().cuda_stream)
    assert st == 580, st
    return {"lse": lse, "ce": ce, "scalars": sc, "grad_logits": g}


def _rel_l2(a, b):
    a, b = a.double(), b.double()
    return float(torch.linalg.norm(a - b) / torch.linalg.norm(b))


def _close(a, b, tol):
    a, b = a.double(), b.double()
    return bool(((a - b).abs() / torch.clamp(b.abs(), min=1.0) <= tol).all())


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_static_matches_workspace_entry_point_twice(L, dtype):
    lt, gt = (BF16_LOSS, BF16_GRAD) if dtype == torch.bfloat16 else (F32_LOSS, F32_GRAD)
    g = torch.Generator(device="cuda").manual_seed(7)
    cases = [(300, 4099, None, 0.0, 1.0), (1000, 32000, 0.1, 1e-3, 2.5)]
    for n, V, mfrac, wz, gs in cases:          # two calls in a row, different shapes
        X = (torch.randn(n, V, device="cuda", generator=g) * 2).to(dtype)
        y = torch.randint(0, V, (n,), device="cuda", generator=g)
        m = None
        if mfrac:
            m = (torch.rand(n, device="cuda", generator=g) > mfrac).to(torch.uint8)
        s = _call_static(L, X, y, m, wz, gs)
        r = L.lossk_ce_from_logits(X, y, loss_mask=m, z_weight=wz, grad_scale=gs, want_grad=True)
        torch.cuda.synchronize()
        for k in ("lse", "ce", "scalars"):
            assert _close(s[k], r[k], lt), k
            assert torch.equal(s[k], r[k]), k
        assert _rel_l2(s["grad_logits"], r["grad_logits"]) <= gt
        assert torch.equal(s["grad_logits"], r["grad_logits"])


def test_static_refuses_beyond_its_limit(L):
    n, V = 16385, 8
    X = torch.zeros(n, V, device="cuda")
    y = torch.zeros(n, dtype=torch.int64, device="cuda")
    with pytest.raises(L.LosskError) as e:
        L.lossk_ce_from_logits_static(X, y)
    assert e.value.status == 583
    y[3] = V
    with pytest.raises(L.LosskError) as e:
        L.lossk_ce_from_logits_static(X[:100].contiguous(), y[:100].contiguous())
    assert e.value.status == 586
