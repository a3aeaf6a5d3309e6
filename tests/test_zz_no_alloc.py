"""lossk_ce_from_logits_static: the entry point for callers that cannot allocate.

Some callers (a plug-in whose device memory all belongs to its host framework's
arena, a runtime with a memory plan fixed at start-up) can neither allocate
nor hand the library a workspace.  This entry point keeps its scratch in a
device array built into the library.  The test calls it through the C ABI
twice in a row, on different inputs, and checks each result against the
fp64 oracle and against the workspace-based lossk_ce_from_logits (the
kernels being the same, for identical bits), in bf16, fp16 and fp32.  It runs
last so that a failure here leaves every other test already run; it must pass
both in a fresh process and after the rest of the suite.
"""
import numpy as np
import pytest
import torch

import lossk_inputs as li
import oracle

pytestmark = pytest.mark.gpu

BF16_LOSS, BF16_GRAD = 2e-3, 1e-2
F32_LOSS, F32_GRAD = 1e-6, 1e-5
DTYPES = {"bf16": torch.bfloat16, "f16": torch.float16, "fp32": torch.float32}
CODES = {"fp32": 0, "bf16": 1, "f16": 2}


@pytest.fixture(scope="module")
def L():
    from conftest import build_lib
    build_lib()
    import output_projection_cross_gb300 as L
    assert torch.cuda.is_available()
    return L


def _call_static(L, X, y, mask, wz, gs, code):
    """Through the C ABI directly: every output allocated here, before the call."""
    n, V = X.shape
    lse = torch.empty(n, dtype=torch.float32, device="cuda")
    ce = torch.empty(n, dtype=torch.float32, device="cuda")
    sc = torch.empty(3, dtype=torch.float64, device="cuda")
    g = torch.empty_like(X)
    st = L.lib.lossk_ce_from_logits_static(
        n, V, code, X.data_ptr(), X.numel(), y.data_ptr(), y.numel(),
        None if mask is None else mask.data_ptr(), wz, gs, lse.data_ptr(), ce.data_ptr(),
        sc.data_ptr(), g.data_ptr(), g.numel(), torch.cuda.current_stream().cuda_stream)
    assert st == 580, st
    return {"lse": lse, "ce": ce, "scalars": sc, "grad_logits": g}


def _rel_l2(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def _close(got, ref, tol, relative):
    """fp32: |d| <= tol |ref| (absolute only where ref is 0); 16-bit: |d| <= tol max(1, |ref|)."""
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    scale = np.where(ref == 0, 1.0, np.abs(ref)) if relative else np.maximum(1.0, np.abs(ref))
    return bool((np.abs(got - ref) / scale <= tol).all())


def _np(t):
    return t.detach().double().cpu().numpy()


@pytest.mark.parametrize("dtype", ["bf16", "f16", "fp32"])
def test_static_matches_oracle_and_workspace_entry_point_twice(L, dtype):
    f32 = dtype == "fp32"
    lt, gt = (F32_LOSS, F32_GRAD) if f32 else (BF16_LOSS, BF16_GRAD)
    cases = [(300, 4099, 0.0, 0.0, 1.0), (1000, 32000, 0.1, 1e-3, 2.5)]
    for i, (n, V, mfrac, wz, gs) in enumerate(cases):      # two calls in a row, different shapes
        g = np.random.default_rng(70 + i)
        Xn = li.round_to((g.standard_normal((n, V)) * 2).astype(np.float32), dtype)
        yn = g.integers(0, V, n).astype(np.int64)
        mn = li.mask(5 + i, n, mfrac) if mfrac else None
        X = torch.from_numpy(Xn).cuda().to(DTYPES[dtype])
        y = torch.from_numpy(yn).cuda()
        m = None if mn is None else torch.from_numpy(mn).cuda()
        before = L.lossk_launch_count()
        s = _call_static(L, X, y, m, wz, gs, CODES[dtype])
        n_static = L.lossk_launch_count() - before
        before = L.lossk_launch_count()
        r = L.lossk_ce_from_logits(X, y, loss_mask=m, z_weight=wz, grad_scale=gs, want_grad=True)
        n_ws = L.lossk_launch_count() - before
        torch.cuda.synchronize()
        # every kernel of the call is counted, as for the workspace entry point
        assert n_static == n_ws and n_static >= 3, (n_static, n_ws)
        ref = oracle.ce_from_logits(Xn, yn, mask=mn, z_weight=wz, grad_scale=gs, want_grad=True)
        assert _close(_np(s["lse"]), ref["lse"], lt, f32)
        assert _close(_np(s["ce"]), ref["ce"], lt, f32)
        assert _close(_np(s["scalars"]), [ref["total"], ref["ce_mean"], ref["z_mean"]], lt, f32)
        # an fp16 gradient is held to the exact gradient rounded to fp16 (its
        # elements lie in fp16's subnormal range at these vocabularies)
        gref = li.round_to(ref["grad"], "f16") if dtype == "f16" else ref["grad"]
        assert _rel_l2(_np(s["grad_logits"]), gref) <= gt
        for k in ("lse", "ce", "scalars", "grad_logits"):
            assert torch.equal(s[k], r[k]), k


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
