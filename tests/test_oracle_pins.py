"""Pins for the fp64 oracle: each test ties it to something other than itself.

Kinds of pin used here:
  * values the pages print (tests/golden/*.json, each with its citation);
  * closed forms (uniform logits -> log V, z = lse^2, zero-gradient cases);
  * invariants the pages state (bit-exact chunk invariance; d_weight summed
    over the vocabulary cancels);
  * library routines in float64 (torch.nn.functional.cross_entropy,
    log_softmax, logsumexp, and torch.autograd for every gradient);
  * central finite differences (the pages' own gradient check);
  * a pure-Python brute force on tiny inputs.
A plausible slip in the oracle -- a dropped z term, a wrong sign, a
transposed operand, a wrong divisor, a chunk-dependent sum -- fails at
least one of these.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute

F64 = torch.float64


def _rand(seed, n, d, V, hs=1.0, ws=0.3):
    g = np.random.default_rng(seed)
    H = g.standard_normal((n, d)).astype(np.float32) * np.float32(hs)
    W = g.standard_normal((V, d)).astype(np.float32) * np.float32(ws)
    y = g.integers(0, V, n).astype(np.int64)
    return H, W, y


def _torch_ce_total(H, W, y, mask, wz):
    """Mean over unmasked tokens of ce + wz*lse^2, via torch library calls."""
    logits = H @ W.T
    ce = torch.nn.functional.cross_entropy(logits, y, reduction="none")
    lse = torch.logsumexp(logits, dim=1)
    m = torch.ones_like(ce) if mask is None else mask
    nv = m.sum()
    return ((ce + wz * lse * lse) * m).sum() / nv, ce, lse


# ---- contract: printed values ----------------------------------------------

def test_status_names(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "status_codes.json")))
    for code, name in g["names"].items():
        assert oracle.status_name(int(code)) == name
    for code in g["unknown"]:
        assert oracle.status_name(code) == "unknown_status"


def test_peak_and_budget_goldens(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "peak_logit_cells.json")))
    for c in g["peak_cases"]:
        r = oracle.peak_logit_cells(c["n_tok"], c["vocab"], c["chunk"])
        for k in ("chunked_cells", "materialized_cells", "ratio", "n_chunks", "status"):
            assert r[k] == c[k], k
    for c in g["dims_cases"]:
        assert oracle.dims_check(c["n_tok"], c["d_model"], c["vocab"]) == c["status"]
    for c in g["chunk_cases"]:
        assert oracle.chunk_check(c["chunk"], c["vocab"]) == c["status"]
    # 2048*151936 is 2.3x the logit-cell ceiling (printed ratio, one decimal)
    assert round(2048 * 151936 / g["constants"]["LOSS_MAX_LOGIT_CELLS"], 1) == 2.3
    assert 2048 * 4096 * 151936 <= g["constants"]["LOSS_MAX_WORK_CELLS"]


def test_budget_edges():
    # work budget: exactly 2^46 fits, one more cell does not
    assert oracle.work_fits(1 << 16, 1 << 15, 1 << 15, 1 << 46)
    assert not oracle.work_fits((1 << 16) + 1, 1 << 15, 1 << 15, 1 << 46)
    assert oracle.dims_check(1 << 16, 1 << 15, 1 << 15) == 580
    assert oracle.dims_check((1 << 16) + 1, 1 << 15, 1 << 15) == 584
    # no overflow in the check itself: a product far past 2^63
    assert not oracle.work_fits(1 << 24, 1 << 24, 1 << 24, 1 << 46)
    # chunk budget: chunk*V == 2^27 exactly passes, one more row refuses
    assert oracle.chunk_check(1 << 10, 1 << 17) == 580
    assert oracle.chunk_check((1 << 10) + 1, 1 << 17) == 587
    # empty and too-large dimensions
    assert oracle.dims_check(0, 4, 4) == 581
    assert oracle.dims_check(4, 0, 4) == 581
    assert oracle.dims_check(4, 4, -3) == 581
    assert oracle.dims_check((1 << 24) + 1, 1, 1) == 583
    assert oracle.chunk_check(0, 10) == 581
    assert oracle.logit_cells(256, 151936) == 38895616.0
    assert oracle.logit_cells(0, 151936) < 0 and oracle.logit_cells(3, -1) < 0
    r = oracle.peak_logit_cells(100, 151936, 2048)      # chunk larger than the batch
    assert r["chunked_cells"] == 100 * 151936 and r["n_chunks"] == 1 and r["status"] == 587
    r = oracle.peak_logit_cells(1000, 10, 3)
    assert r["n_chunks"] == 334 and r["ratio"] == 1000 / 3
    r = oracle.peak_logit_cells(0, 10, 3)
    assert r["status"] == 581 and r["chunked_cells"] < 0 and r["n_chunks"] == 0


def test_target_guard_refuses():
    H, W, y = _rand(0, 5, 3, 11)
    for bad in (-1, 11, 1 << 40):
        yy = y.copy()
        yy[2] = bad
        assert not oracle.targets_in_range(yy, 5, 11)
        with pytest.raises(oracle.OracleError) as e:
            oracle.ce_fwd(H, W, yy, chunk=2)
        assert e.value.status == 586
    # a masked token's target must still be in range (every one of the first n)
    yy = y.copy()
    yy[0] = -1
    m = np.ones(5, np.uint8)
    m[0] = 0
    with pytest.raises(oracle.OracleError) as e:
        oracle.ce_fwd(H, W, yy, mask=m, chunk=2)
    assert e.value.status == 586


def test_scalar_guard_refuses():
    H, W, y = _rand(0, 5, 3, 11)
    for wz in (float("nan"), float("inf"), -1.0):
        with pytest.raises(oracle.OracleError) as e:
            oracle.ce_fwd(H, W, y, chunk=2, z_weight=wz)
        assert e.value.status == 585
    with pytest.raises(oracle.OracleError) as e:
        oracle.ce_bwd(H, W, y, grad_scale=float("nan"))
    assert e.value.status == 585
    T = np.zeros((5, 11), np.float32)
    for temp in (0.0, -1.0, float("inf")):
        with pytest.raises(oracle.OracleError) as e:
            oracle.distill(H, W, T, "ce", temperature=temp)
        assert e.value.status == 585
    with pytest.raises(oracle.OracleError) as e:
        oracle.distill(H, W, T, 3)
    assert e.value.status == 588
    with pytest.raises(oracle.OracleError) as e:
        oracle.ce_fwd(H, W, y, chunk=(1 << 27) // 11 + 1)
    assert e.value.status == 587


# ---- closed forms ------------------------------------------------------------

def test_uniform_logits_ln9_golden(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "uniform_logits_ln9.json")))
    logits = np.full((g["n_tok"], g["vocab"]), g["logit_value"], np.float32)
    r = oracle.ce_from_logits(logits, g["targets"])
    assert r["total"] == g["mean_loss"]            # to the last bit
    assert r["total"] == math.log(9)


@pytest.mark.parametrize("V", [9, 1000, 151936])
def test_zero_weight_gives_log_vocab(V):
    n, d = 6, 5
    H = np.random.default_rng(1).standard_normal((n, d)).astype(np.float32)
    W = np.zeros((V, d), np.float32)
    y = np.random.default_rng(2).integers(0, V, n)
    for chunk in (1, 4, n):
        r = oracle.ce_fwd(H, W, y, chunk=chunk, z_weight=0.5)
        assert r["ce_mean"] == math.log(V)
        assert np.all(r["lse"] == math.log(V))
        assert r["z_mean"] == pytest.approx(math.log(V) ** 2, rel=1e-15)
        assert r["total"] == pytest.approx(math.log(V) + 0.5 * math.log(V) ** 2, rel=1e-15)


def test_vocab_of_one_closed_form():
    """One class: the softmax is 1, so CE = lse - s_y = 0 and its gradient
    vanishes; what remains is the z term, z = lse^2 = s^2, with d(loss)/ds =
    a 2 w_z lse (a = grad_scale / n)."""
    n, d, wz, gs = 5, 8, 0.05, 0.75
    g = np.random.default_rng(61)
    H = g.standard_normal((n, d)).astype(np.float32)
    W = (g.standard_normal((1, d)) * 0.3).astype(np.float32)
    y = np.zeros(n, np.int64)
    r = oracle.ce_fwd(H, W, y, z_weight=wz)
    dH, dW = oracle.ce_bwd(H, W, y, z_weight=wz, grad_scale=gs)
    s = H.astype(np.float64) @ W.astype(np.float64).T          # [n][1]
    assert np.all(r["ce"] == 0.0)
    assert np.allclose(r["lse"], s[:, 0], rtol=0, atol=1e-12)
    assert np.isclose(r["z_mean"], np.mean(s[:, 0] ** 2), rtol=1e-12)
    gl = (gs / n) * 2 * wz * s                                   # d(loss)/ds, [n][1]
    assert np.allclose(dH, gl * W.astype(np.float64), rtol=1e-10, atol=1e-14)
    assert np.allclose(dW, gl.T @ H.astype(np.float64), rtol=1e-10, atol=1e-14)


def test_z_is_lse_squared():
    H, W, y = _rand(3, 7, 4, 13)
    r = oracle.ce_fwd(H, W, y, chunk=3, z_weight=0.25)
    assert r["z_mean"] == pytest.approx(np.mean(r["lse"] ** 2), rel=1e-14)
    assert r["total"] == pytest.approx(r["ce_mean"] + 0.25 * r["z_mean"], rel=1e-14)


# ---- invariants the pages state --------------------------------------------

def test_chunk_invariance_every_chunk_bit_exact():
    H, W, y = _rand(4, 12, 6, 37)
    base = oracle.ce_fwd(H, W, y, chunk=12, z_weight=0.1)
    for chunk in range(1, 13):
        r = oracle.ce_fwd(H, W, y, chunk=chunk, z_weight=0.1)
        assert r["total"] == base["total"]
        assert np.array_equal(r["lse"], base["lse"])
        assert np.array_equal(r["ce"], base["ce"])


def test_chunk_invariance_larger():
    H, W, y = _rand(5, 300, 32, 2000, ws=0.05)
    base = oracle.ce_fwd(H, W, y, chunk=300)
    for chunk in (1, 16, 256):
        r = oracle.ce_fwd(H, W, y, chunk=chunk)
        assert r["total"] == base["total"] and np.array_equal(r["lse"], base["lse"])


def test_dweight_vocab_sum_cancels():
    # [P1] backward section: summing d_weight over the vocabulary cancels to
    # within 1e-9 (softmax and the one-hot both sum to one).
    H, W, y = _rand(6, 16, 8, 300)
    dH, dW = oracle.ce_bwd(H, W, y)
    assert np.abs(dW.sum(axis=0)).max() <= 1e-9
    # with z-loss the row sum of G is alpha*2*wz*lse_t, so the cancellation
    # leaves sum_t alpha*2*wz*lse_t*H_t
    wz = 0.3
    dH, dW = oracle.ce_bwd(H, W, y, z_weight=wz)
    lse = oracle.ce_fwd(H, W, y, chunk=16)["lse"]
    expect = (2 * wz * lse / 16)[:, None] * H.astype(np.float64)
    assert np.allclose(dW.sum(axis=0), expect.sum(axis=0), atol=1e-12, rtol=1e-10)


# ---- library routines in float64 -------------------------------------------

@pytest.mark.parametrize("seed", [0, 1])
def test_ce_matches_torch_library(seed):
    H, W, y = _rand(seed, 20, 7, 53)
    mask = np.random.default_rng(seed + 9).integers(0, 2, 20).astype(np.uint8)
    mask[0] = 1
    wz, gs = 0.2, 1.7
    r = oracle.ce_fwd(H, W, y, mask=mask, chunk=6, z_weight=wz)
    Ht = torch.tensor(H, dtype=torch.float64, requires_grad=True)
    Wt = torch.tensor(W, dtype=torch.float64, requires_grad=True)
    tot, ce, lse = _torch_ce_total(Ht, Wt, torch.tensor(y), torch.tensor(mask, dtype=torch.float64), wz)
    assert r["total"] == pytest.approx(tot.item(), rel=1e-13)
    assert np.allclose(r["lse"], lse.detach().numpy(), rtol=1e-13, atol=0)
    assert np.allclose(r["ce"], (ce * torch.tensor(mask)).detach().numpy(), rtol=1e-12, atol=1e-14)
    (gs * tot).backward()
    dH, dW = oracle.ce_bwd(H, W, y, mask=mask, z_weight=wz, grad_scale=gs)
    assert np.allclose(dH, Ht.grad.numpy(), rtol=1e-11, atol=1e-15)
    assert np.allclose(dW, Wt.grad.numpy(), rtol=1e-11, atol=1e-15)


def test_ce_from_logits_matches_torch_library():
    g = np.random.default_rng(7)
    X = (g.standard_normal((9, 31)) * 3).astype(np.float32)
    y = g.integers(0, 31, 9)
    mask = np.array([1, 1, 0, 1, 1, 1, 0, 1, 1], np.uint8)
    wz, gs = 0.05, 0.5
    r = oracle.ce_from_logits(X, y, mask=mask, z_weight=wz, grad_scale=gs, want_grad=True)
    Xt = torch.tensor(X, dtype=torch.float64, requires_grad=True)
    ce = torch.nn.functional.cross_entropy(Xt, torch.tensor(y), reduction="none")
    lse = torch.logsumexp(Xt, 1)
    m = torch.tensor(mask, dtype=torch.float64)
    tot = ((ce + wz * lse ** 2) * m).sum() / m.sum()
    (gs * tot).backward()
    assert r["total"] == pytest.approx(tot.item(), rel=1e-13)
    assert np.allclose(r["grad"], Xt.grad.numpy(), rtol=1e-11, atol=1e-16)


# ---- finite differences (the pages' own gradient check) --------------------

def _fd(f, x, h=1e-6):
    g = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        g[idx] = (f(xp) - f(xm)) / (2 * h)
    return g


def _total_from_f64(H, W, y, mask, wz):
    # the fp32 input boundary would round H+h; use the pure-Python brute force,
    # which takes Python floats, to evaluate the loss at perturbed points.
    return brute.ce(H.tolist(), W.tolist(), list(y), None if mask is None else list(mask), wz)[0]


@pytest.mark.parametrize("wz", [0.0, 0.3])
def test_ce_grad_central_difference(wz):
    n, d, V = 4, 3, 7
    g = np.random.default_rng(11)
    H = g.standard_normal((n, d)).astype(np.float32)
    W = g.standard_normal((V, d)).astype(np.float32)
    y = g.integers(0, V, n)
    mask = np.array([1, 0, 1, 1], np.uint8)
    dH, dW = oracle.ce_bwd(H, W, y, mask=mask, z_weight=wz)
    H64, W64 = H.astype(np.float64), W.astype(np.float64)
    fdH = _fd(lambda x: _total_from_f64(x, W64, y, mask, wz), H64)
    fdW = _fd(lambda x: _total_from_f64(H64, x, y, mask, wz), W64)
    assert np.abs(dH - fdH).max() <= 1e-8
    assert np.abs(dW - fdW).max() <= 1e-8


# ---- brute force ------------------------------------------------------------

@pytest.mark.parametrize("shape", [(1, 1, 2), (3, 5, 7), (8, 8, 50)])
def test_ce_brute_force(shape):
    n, d, V = shape
    H, W, y = _rand(sum(shape), n, d, V)
    mask = (np.arange(n) % 3 != 1).astype(np.uint8)
    wz, gs = 0.07, 2.0
    tot, lses, bdH, bdW = brute.ce(H.astype(np.float64).tolist(), W.astype(np.float64).tolist(),
                                   list(y), list(mask), wz, gs)
    r = oracle.ce_fwd(H, W, y, mask=mask, chunk=2, z_weight=wz)
    dH, dW = oracle.ce_bwd(H, W, y, mask=mask, z_weight=wz, grad_scale=gs)
    assert r["total"] == pytest.approx(tot, rel=1e-12)
    assert np.allclose(r["lse"], lses, rtol=1e-12)
    assert np.allclose(dH, bdH, rtol=1e-10, atol=1e-15)
    assert np.allclose(dW, bdW, rtol=1e-10, atol=1e-15)


# ---- masking ----------------------------------------------------------------

def test_masked_tokens_do_not_count():
    H, W, y = _rand(12, 10, 4, 29)
    mask = np.array([1, 1, 0, 1, 0, 1, 1, 1, 1, 0], np.uint8)
    r1 = oracle.ce_fwd(H, W, y, mask=mask, chunk=3, z_weight=0.1)
    H2 = H.copy()
    H2[mask == 0] = 5.0                      # change only the masked rows
    y2 = y.copy()
    y2[mask == 0] = 0
    r2 = oracle.ce_fwd(H2, W, y2, mask=mask, chunk=3, z_weight=0.1)
    assert r1["total"] == r2["total"]
    assert np.all(r1["ce"][mask == 0] == 0)
    dH, dW = oracle.ce_bwd(H, W, y, mask=mask, z_weight=0.1)
    assert np.all(dH[mask == 0] == 0)
    # the divisor is the number of counted tokens: repeating a counted token's
    # row as an extra masked token changes nothing
    keep = mask == 1
    r3 = oracle.ce_fwd(H[keep], W, y[keep], chunk=3, z_weight=0.1)
    assert r3["total"] == pytest.approx(r1["total"], rel=1e-14)
    # nothing counted: zeros, still status ok
    z = oracle.ce_fwd(H, W, y, mask=np.zeros(10, np.uint8), chunk=3)
    assert z["total"] == 0.0
    dH, dW = oracle.ce_bwd(H, W, y, mask=np.zeros(10, np.uint8))
    assert not dH.any() and not dW.any()


def test_superposition_in_z_weight():
    H, W, y = _rand(13, 9, 5, 40)
    r0 = oracle.ce_fwd(H, W, y, chunk=4)
    r1 = oracle.ce_fwd(H, W, y, chunk=4, z_weight=0.01)
    assert r1["total"] == pytest.approx(r0["total"] + 0.01 * r0["z_mean"], rel=1e-14)
    a0, b0 = oracle.ce_bwd(H, W, y)
    a1, b1 = oracle.ce_bwd(H, W, y, z_weight=1.0)
    a2, b2 = oracle.ce_bwd(H, W, y, z_weight=0.5)
    assert np.allclose(a2, a0 + 0.5 * (a1 - a0), rtol=1e-12, atol=1e-15)
    assert np.allclose(b2, b0 + 0.5 * (b1 - b0), rtol=1e-12, atol=1e-15)


# ---- distillation -------------------------------------------------------------

def _torch_distill(H, W, Tt, direction, T, mask, wz):
    a = torch.log_softmax(H @ W.T / T, dim=1)
    lp = torch.log_softmax(Tt / T, dim=1)
    if direction == "ce":
        L = -(lp.exp() * a).sum(1)
    elif direction == "fkl":
        L = torch.nn.functional.kl_div(a, lp, reduction="none", log_target=True).sum(1)
    else:
        L = torch.nn.functional.kl_div(lp, a, reduction="none", log_target=True).sum(1)
    lse = torch.logsumexp(H @ W.T / T, dim=1)
    m = torch.ones(H.shape[0], dtype=F64) if mask is None else torch.tensor(mask, dtype=F64)
    return ((L + wz * lse * lse) * m).sum() / m.sum(), L


@pytest.mark.parametrize("direction", ["ce", "fkl", "rkl"])
@pytest.mark.parametrize("T,wz", [(1.0, 0.0), (2.0, 0.1), (0.7, 0.0)])
def test_distill_matches_torch_library(direction, T, wz):
    H, W, _ = _rand(20, 11, 6, 45)
    Tt = (np.random.default_rng(21).standard_normal((11, 45)) * 3).astype(np.float32)
    mask = np.array([1, 1, 1, 0, 1, 1, 1, 1, 0, 1, 1], np.uint8)
    gs = 1.3
    r = oracle.distill(H, W, Tt, direction, temperature=T, mask=mask, chunk=4, z_weight=wz,
                       grad_scale=gs)
    Ht = torch.tensor(H, dtype=torch.float64, requires_grad=True)
    Wt = torch.tensor(W, dtype=torch.float64, requires_grad=True)
    tot, L = _torch_distill(Ht, Wt, torch.tensor(Tt, dtype=torch.float64), direction, T, mask, wz)
    assert r["total"] == pytest.approx(tot.item(), rel=1e-12)
    assert np.allclose(r["per_token"], L.detach().numpy() * mask, rtol=1e-10, atol=1e-13)
    (gs * tot).backward()
    assert np.allclose(r["dH"], Ht.grad.numpy(), rtol=1e-10, atol=1e-14)
    assert np.allclose(r["dW"], Wt.grad.numpy(), rtol=1e-10, atol=1e-14)


def _torch_distill_logits(X, Tt, direction, T, mask, wz, reduce_sum):
    """The three objectives written with torch's own log_softmax / kl_div /
    logsumexp, on given student logits X (the from-distribution form)."""
    a = torch.log_softmax(X / T, dim=1)
    lp = torch.log_softmax(Tt / T, dim=1)
    if direction == "ce":
        L = -(lp.exp() * a).sum(1)
    elif direction == "fkl":
        L = torch.nn.functional.kl_div(a, lp, reduction="none", log_target=True).sum(1)
    else:
        L = torch.nn.functional.kl_div(lp, a, reduction="none", log_target=True).sum(1)
    lse = torch.logsumexp(X / T, dim=1)
    m = torch.ones(X.shape[0], dtype=F64) if mask is None else torch.tensor(mask, dtype=F64)
    s = ((L + wz * lse * lse) * m).sum()
    return (s if reduce_sum else s / m.sum()), L, lse


@pytest.mark.parametrize("direction", ["ce", "fkl", "rkl"])
@pytest.mark.parametrize("T,wz,reduce_sum", [(1.0, 0.0, False), (2.0, 0.1, False), (0.7, 0.05, True)])
def test_distill_from_logits_matches_torch_library(direction, T, wz, reduce_sum):
    g = np.random.default_rng(22)
    X = g.standard_normal((9, 37)).astype(np.float32) * 2
    Tt = (g.standard_normal((9, 37)) * 3).astype(np.float32)
    mask = np.array([1, 0, 1, 1, 1, 1, 0, 1, 1], np.uint8)
    gs = 0.8
    r = oracle.distill_from_logits(X, Tt, direction, temperature=T, mask=mask, z_weight=wz,
                                   grad_scale=gs, reduce_sum=reduce_sum)
    Xt = torch.tensor(X, dtype=F64, requires_grad=True)
    tot, L, lse = _torch_distill_logits(Xt, torch.tensor(Tt, dtype=F64), direction, T, mask, wz,
                                        reduce_sum)
    assert r["total"] == pytest.approx(tot.item(), rel=1e-12)
    assert np.allclose(r["per_token"], L.detach().numpy() * mask, rtol=1e-10, atol=1e-13)
    assert np.allclose(r["lse"], lse.detach().numpy(), rtol=1e-13)
    (gs * tot).backward()
    assert np.allclose(r["grad"], Xt.grad.numpy(), rtol=1e-10, atol=1e-14)


def test_distill_from_logits_sum_is_mean_times_count():
    g = np.random.default_rng(23)
    X = g.standard_normal((7, 20)).astype(np.float32)
    Tt = g.standard_normal((7, 20)).astype(np.float32)
    mask = np.array([1, 1, 0, 1, 1, 0, 1], np.uint8)
    a = oracle.distill_from_logits(X, Tt, "fkl", temperature=1.5, mask=mask, z_weight=0.1)
    b = oracle.distill_from_logits(X, Tt, "fkl", temperature=1.5, mask=mask, z_weight=0.1,
                                   reduce_sum=True)
    assert b["total"] == pytest.approx(a["total"] * 5, rel=1e-14)
    assert np.allclose(b["grad"], a["grad"] * 5, rtol=1e-13, atol=1e-16)


def test_distill_uniform_teacher_zero_weight():
    n, d, V = 5, 4, 17
    H = np.random.default_rng(3).standard_normal((n, d)).astype(np.float32)
    W = np.zeros((V, d), np.float32)
    Tt = np.full((n, V), 1.5, np.float32)
    for direction in ("ce", "fkl", "rkl"):
        r = oracle.distill(H, W, Tt, direction, temperature=2.0)
        if direction == "ce":
            assert r["total"] == pytest.approx(math.log(V), rel=1e-15)
        else:
            assert abs(r["total"]) <= 1e-15
        assert np.abs(r["dH"]).max() <= 1e-16 and np.abs(r["dW"]).max() <= 1e-16


def test_distill_one_hot_teacher_is_label_ce():
    H, W, y = _rand(30, 8, 5, 23)
    Tt = np.full((8, 23), -60.0, np.float32)
    Tt[np.arange(8), y] = 60.0
    r = oracle.distill(H, W, Tt, "ce", temperature=1.0)
    c = oracle.ce_fwd(H, W, y, chunk=8)
    assert r["total"] == pytest.approx(c["total"], rel=1e-12)
    dH, dW = oracle.ce_bwd(H, W, y)
    assert np.allclose(r["dH"], dH, rtol=1e-9, atol=1e-14)
    assert np.allclose(r["dW"], dW, rtol=1e-9, atol=1e-14)


def test_distill_kl_identities():
    H, W, _ = _rand(31, 9, 5, 33)
    Tt = (np.random.default_rng(32).standard_normal((9, 33)) * 3).astype(np.float32)
    T = 2.0
    ce = oracle.distill(H, W, Tt, "ce", temperature=T)
    fkl = oracle.distill(H, W, Tt, "fkl", temperature=T)
    rkl = oracle.distill(H, W, Tt, "rkl", temperature=T)
    # fKL = CE - H(p), with the teacher entropy from a library routine
    lp = torch.log_softmax(torch.tensor(Tt, dtype=torch.float64) / T, 1)
    ent = -(lp.exp() * lp).sum(1).numpy()
    assert np.allclose(fkl["per_token"], ce["per_token"] - ent, rtol=1e-12, atol=1e-13)
    # CE and fKL differ by a constant in the student: same gradients
    assert np.allclose(fkl["dH"], ce["dH"], rtol=1e-12, atol=1e-16)
    assert np.allclose(fkl["dW"], ce["dW"], rtol=1e-12, atol=1e-16)
    assert np.all(rkl["per_token"] >= -1e-15) and np.all(fkl["per_token"] >= -1e-15)


def test_distill_temperature_scaling_identity():
    # distill(H, W, t, T) == distill(H/T, W, t/T, 1) for the losses; T = 2 keeps
    # the scaled inputs exact.
    H, W, _ = _rand(33, 7, 6, 29)
    Tt = (np.random.default_rng(34).standard_normal((7, 29)) * 3).astype(np.float32)
    for direction in ("ce", "fkl", "rkl"):
        a = oracle.distill(H, W, Tt, direction, temperature=2.0, z_weight=0.1, want_grad=False)
        b = oracle.distill(H / 2, W, Tt / 2, direction, temperature=1.0, z_weight=0.1,
                           want_grad=False)
        assert a["total"] == b["total"]
        assert np.array_equal(a["per_token"], b["per_token"])


@pytest.mark.parametrize("direction", ["ce", "fkl", "rkl"])
def test_distill_masked_vocabulary_is_the_smaller_vocabulary(direction):
    """Vocabulary entries masked out (-inf) in both the student and the teacher
    row have probability 0 in both: the losses, lse and the gradient on the kept
    entries equal those over the kept entries alone, and the gradient is 0 on
    the masked ones."""
    n, V, T, wz = 5, 23, 1.5, 0.1
    g = np.random.default_rng(64)
    X = (g.standard_normal((n, V)) * 2).astype(np.float32)
    Tt = (g.standard_normal((n, V)) * 3).astype(np.float32)
    drop = np.array([0, 4, 5, 6, 13, 22])
    keep = np.setdiff1d(np.arange(V), drop)
    Xm, Tm = X.copy(), Tt.copy()
    Xm[:, drop] = -np.inf
    Tm[:, drop] = -np.inf
    a = oracle.distill_from_logits(Xm, Tm, direction, temperature=T, z_weight=wz)
    b = oracle.distill_from_logits(X[:, keep], Tt[:, keep], direction, temperature=T, z_weight=wz)
    assert np.allclose(a["per_token"], b["per_token"], rtol=1e-12, atol=1e-13)
    assert np.allclose(a["lse"], b["lse"], rtol=1e-12, atol=1e-13)
    assert np.isclose(a["total"], b["total"], rtol=1e-12)
    assert np.allclose(a["grad"][:, keep], b["grad"], rtol=1e-12, atol=1e-15)
    assert np.all(a["grad"][:, drop] == 0.0)


@pytest.mark.parametrize("direction", ["ce", "fkl", "rkl"])
@pytest.mark.parametrize("side", ["teacher", "student"])
def test_distill_one_sided_mask_is_the_limit(direction, side):
    """Entries masked out (-inf) on one side only give the limit of a logit going
    to -inf there.  Where the masked side's probability only weights the term
    (teacher zeros in CE and forward KL, student zeros in reverse KL), the -inf
    result equals that at a finite logit far enough down for exp to underflow
    to 0.  Where the other side keeps mass on a masked entry (student zeros in
    CE and forward KL, teacher zeros in reverse KL), the loss is +inf: the
    finite stand-ins grow in proportion to the logit's depth."""
    n, V, T, wz = 4, 19, 1.5, 0.1
    g = np.random.default_rng(71)
    X = (g.standard_normal((n, V)) * 2).astype(np.float32)
    Tt = (g.standard_normal((n, V)) * 3).astype(np.float32)
    drop = np.array([2, 3, 11])

    def run(value):
        Xm, Tm = X.copy(), Tt.copy()
        (Tm if side == "teacher" else Xm)[:, drop] = value
        return oracle.distill_from_logits(Xm, Tm, direction, temperature=T, z_weight=wz)

    a, far, farther = run(-np.inf), run(-3000.0), run(-6000.0)
    infinite = (side == "student") == (direction != "rkl")
    if infinite:
        assert np.all(np.isposinf(a["per_token"])) and np.isposinf(a["total"])
        # the masked terms grow in proportion to the logit's depth: doubling it
        # nearly doubles the loss
        assert np.all(np.isfinite(far["per_token"])) and np.all(farther["per_token"] > 1.5 * far["per_token"])
    else:
        assert np.all(np.isfinite(a["per_token"]))
        assert np.allclose(a["per_token"], far["per_token"], rtol=1e-12, atol=1e-13)
        assert np.allclose(a["lse"], far["lse"], rtol=1e-12, atol=1e-13)
        assert np.allclose(a["grad"], far["grad"], rtol=1e-12, atol=1e-15)
        if side == "student":
            assert np.all(a["grad"][:, drop] == 0.0)


@pytest.mark.parametrize("direction", ["fkl", "rkl"])
def test_distill_identical_teacher_is_zero(direction):
    """Teacher = student: both KL directions are zero and their gradient is the
    z term's alone, 2 w_z lse q / T per token (mean over the counted tokens)."""
    n, V, T, wz = 6, 11, 1.7, 0.2
    X = (np.random.default_rng(63).standard_normal((n, V)) * 2).astype(np.float32)
    r = oracle.distill_from_logits(X, X, direction, temperature=T, z_weight=wz)
    assert np.allclose(r["per_token"], 0.0, rtol=0, atol=1e-12)
    a = X.astype(np.float64) / T
    lse = np.log(np.exp(a - a.max(1, keepdims=True)).sum(1)) + a.max(1)
    q = np.exp(a - lse[:, None])
    assert np.allclose(r["grad"], (1.0 / n) * 2 * wz * lse[:, None] * q / T, rtol=1e-10, atol=1e-14)


@pytest.mark.parametrize("T", [0.5, 2.0, 3.0])
@pytest.mark.parametrize("direction", ["ce", "fkl", "rkl"])
def test_distill_two_class_closed_form(T, direction):
    """Absolute distillation values at T != 1 by hand.  Student logits (0, T ln 3)
    and teacher logits (0, 0) give q = softmax(s/T) = (1/4, 3/4) and p = (1/2, 1/2)
    exactly, so every loss, lse, z term and gradient is a log of small rationals:
      CE  = -(1/2 ln 1/4 + 1/2 ln 3/4) = ln 4 - 1/2 ln 3
      fKL = 1/2 ln(1/2 / 1/4) + 1/2 ln(1/2 / 3/4) = 1/2 ln 4/3
      rKL = 1/4 ln(1/4 / 1/2) + 3/4 ln(3/4 / 1/2) = 1/4 ln 1/2 + 3/4 ln 3/2
      lse(s/T) = ln(1 + 3) = ln 4, z = (ln 4)^2
    gradients with respect to s: (q - p)/T for CE and fKL,
    q_i (ln q_i - ln p_i - rKL)/T for rKL, plus 2 w_z lse q / T for the z term."""
    X = np.array([[0.0, T * math.log(3.0)]], dtype=np.float64)
    Tt = np.zeros((1, 2))
    wz = 0.3
    r = oracle.distill_from_logits(X, Tt, direction, temperature=T, z_weight=wz)
    q, pt = np.array([0.25, 0.75]), np.array([0.5, 0.5])
    L = {"ce": math.log(4) - 0.5 * math.log(3), "fkl": 0.5 * math.log(4 / 3),
         "rkl": 0.25 * math.log(0.5) + 0.75 * math.log(1.5)}[direction]
    lse = math.log(4)
    if direction == "rkl":
        g = q * (np.log(q) - np.log(pt) - L) / T
    else:
        g = (q - pt) / T
    g = g + 2 * wz * lse * q / T
    # the student logit T ln 3 goes through fp32 in the oracle's interface:
    # about 1e-7 relative, far below these bounds
    assert abs(r["per_token"][0] - L) <= 1e-6
    assert abs(r["lse"][0] - lse) <= 1e-6
    assert abs(r["distill_mean"] - L) <= 1e-6
    assert abs(r["z_mean"] - lse * lse) <= 1e-6
    assert abs(r["total"] - (L + wz * lse * lse)) <= 1e-6
    assert np.allclose(r["grad"][0], g, rtol=0, atol=1e-6)


@pytest.mark.parametrize("direction", ["ce", "fkl", "rkl"])
@pytest.mark.parametrize("wz", [0.0, 0.2])
def test_distill_grad_central_difference(direction, wz):
    n, d, V = 3, 3, 6
    g = np.random.default_rng(40)
    H = g.standard_normal((n, d)).astype(np.float32)
    W = g.standard_normal((V, d)).astype(np.float32)
    Tt = (g.standard_normal((n, V)) * 2).astype(np.float32)
    T = 1.5
    r = oracle.distill(H, W, Tt, direction, temperature=T, z_weight=wz)
    H64, W64, T64 = H.astype(np.float64), W.astype(np.float64), Tt.astype(np.float64).tolist()

    def tot(Hx, Wx):
        return brute.distill(Hx.tolist(), Wx.tolist(), T64, direction, T, None, wz)[0]

    assert np.abs(r["dH"] - _fd(lambda x: tot(x, W64), H64)).max() <= 1e-8
    assert np.abs(r["dW"] - _fd(lambda x: tot(H64, x), W64)).max() <= 1e-8


@pytest.mark.parametrize("direction", ["ce", "fkl", "rkl"])
def test_distill_brute_force(direction):
    H, W, _ = _rand(50, 6, 4, 19)
    Tt = (np.random.default_rng(51).standard_normal((6, 19)) * 3).astype(np.float32)
    mask = [1, 0, 1, 1, 1, 1]
    tot, per, bdH, bdW = brute.distill(H.astype(np.float64).tolist(), W.astype(np.float64).tolist(),
                                       Tt.astype(np.float64).tolist(), direction, 2.0, mask, 0.05, 0.9)
    r = oracle.distill(H, W, Tt, direction, temperature=2.0, mask=np.array(mask, np.uint8),
                       chunk=2, z_weight=0.05, grad_scale=0.9)
    assert r["total"] == pytest.approx(tot, rel=1e-12)
    assert np.allclose(r["per_token"], per, rtol=1e-10, atol=1e-14)
    assert np.allclose(r["dH"], bdH, rtol=1e-10, atol=1e-15)
    assert np.allclose(r["dW"], bdW, rtol=1e-10, atol=1e-15)


def test_distill_chunk_invariance():
    H, W, _ = _rand(60, 10, 4, 21)
    Tt = (np.random.default_rng(61).standard_normal((10, 21)) * 3).astype(np.float32)
    base = oracle.distill(H, W, Tt, "rkl", temperature=2.0, chunk=10, z_weight=0.1)
    for chunk in range(1, 11):
        r = oracle.distill(H, W, Tt, "rkl", temperature=2.0, chunk=chunk, z_weight=0.1)
        assert r["total"] == base["total"]
        assert np.array_equal(r["dH"], base["dH"]) and np.array_equal(r["dW"], base["dW"])


# ---- sampled-row helpers agree with the whole-tensor oracle -----------------

def test_sampled_rows_match_full():
    H, W, y = _rand(70, 12, 5, 40)
    mask = np.ones(12, np.uint8)
    mask[3] = 0
    wz, gs = 0.1, 1.5
    f = oracle.ce_fwd(H, W, y, mask=mask, chunk=5, z_weight=wz)
    dH, dW = oracle.ce_bwd(H, W, y, mask=mask, z_weight=wz, grad_scale=gs)
    rows = np.array([0, 3, 11])
    s = oracle.ce_token_rows(H, W, y, rows, mask=mask, z_weight=wz, grad_scale=gs)
    assert np.array_equal(s["lse"], f["lse"][rows])
    assert np.allclose(s["dH"], dH[rows], rtol=1e-13, atol=0)
    v = np.array([0, 17, 39])
    dw = oracle.ce_dweight_rows(H, W, y, f["lse"], v, mask=mask, z_weight=wz, grad_scale=gs)
    assert np.allclose(dw, dW[v], rtol=1e-12, atol=1e-16)
    Tt = (np.random.default_rng(71).standard_normal((12, 40)) * 3).astype(np.float32)
    full = oracle.distill(H, W, Tt, "rkl", temperature=2.0, mask=mask, z_weight=wz, grad_scale=gs)
    sd = oracle.distill_token_rows(H, W, Tt, "rkl", rows, temperature=2.0, mask=mask,
                                   z_weight=wz, grad_scale=gs)
    assert np.allclose(sd["loss"][[0, 2]], full["per_token"][rows][[0, 2]], rtol=1e-13)
    assert np.array_equal(sd["lse"], full["lse"][rows])
    assert np.allclose(sd["dH"], full["dH"][rows], rtol=1e-12, atol=1e-17)
    # d_weight rows from every token's lse and loss, all three objectives, with the
    # masked token among the sums (its loss enters nothing)
    for direction in ("ce", "fkl", "rkl"):
        full = oracle.distill(H, W, Tt, direction, temperature=2.0, mask=mask, z_weight=wz,
                              grad_scale=gs)
        allr = oracle.distill_token_rows(H, W, Tt, direction, np.arange(12), temperature=2.0,
                                         mask=mask, z_weight=wz, grad_scale=gs, want_dh=False)
        assert np.array_equal(allr["lse"], full["lse"])
        dwd = oracle.distill_dweight_rows(H, W, Tt, direction, allr["lse"], allr["loss"], v,
                                          temperature=2.0, mask=mask, z_weight=wz, grad_scale=gs)
        assert np.allclose(dwd, full["dW"][v], rtol=1e-11, atol=1e-17), direction
        # the token reduction on its own gives the full oracle's scalars, bit for bit
        r = oracle.reduce_tokens(allr["loss"], allr["lse"], mask=mask, z_weight=wz)
        assert (r["total"], r["loss_mean"], r["z_mean"]) == (full["total"], full["distill_mean"],
                                                             full["z_mean"])
    r = oracle.reduce_tokens(f["ce"], f["lse"], mask=mask, z_weight=wz)
    assert (r["total"], r["loss_mean"], r["z_mean"]) == (f["total"], f["ce_mean"], f["z_mean"])
    assert oracle.reduce_tokens(f["ce"], f["lse"], mask=np.zeros(12, np.uint8))["total"] == 0.0


# ---- vocabulary-parallel cross-entropy ------------------------------------------

def _shards(V, bounds):
    """[(v0, Vs)] for cut points `bounds` inside [0, V)."""
    cuts = [0] + list(bounds) + [V]
    return [(a, b - a) for a, b in zip(cuts[:-1], cuts[1:])]


def test_one_shard_is_the_unsharded_loss_bit_for_bit():
    H, W, y = _rand(81, 9, 6, 33)
    mask = np.ones(9, np.uint8)
    mask[4] = 0
    p = oracle.ce_shard_fwd(H, W, y, 0, 33)
    c = oracle.ce_shard_combine(p[None], mask=mask, z_weight=0.1)
    f = oracle.ce_fwd(H, W, y, mask=mask, z_weight=0.1)
    assert np.array_equal(c["lse"], f["lse"]) and np.array_equal(c["ce"], f["ce"])
    assert (c["total"], c["ce_mean"], c["z_mean"]) == (f["total"], f["ce_mean"], f["z_mean"])
    dh, dw = oracle.ce_shard_bwd(H, W, y, 0, 33, f["lse"], mask=mask, z_weight=0.1, grad_scale=1.5)
    dH, dW = oracle.ce_bwd(H, W, y, mask=mask, z_weight=0.1, grad_scale=1.5)
    assert np.allclose(dh, dH, rtol=1e-13, atol=1e-18) and np.allclose(dw, dW, rtol=1e-13, atol=1e-18)


@pytest.mark.parametrize("bounds", [(16,), (5, 6, 30), (1,), (32,)])
def test_shards_recombine_into_the_unsharded_loss(bounds):
    """Uneven shards, a one-row shard, the target in the first and last rows of
    a shard: the combined loss and the summed (concatenated) gradients are the
    unsharded ones, and the whole-row lse is torch's logsumexp."""
    n, d, V = 12, 7, 33
    H, W, y = _rand(82, n, d, V)
    y[0], y[1], y[2] = 0, V - 1, bounds[0]
    mask = np.ones(n, np.uint8)
    mask[[3, 7]] = 0
    wz, gs = 0.05, 0.7
    parts = np.stack([oracle.ce_shard_fwd(H, W[v0:v0 + vs], y, v0, V) for v0, vs in _shards(V, bounds)])
    assert np.all(parts[:, 2].sum(0) == 1.0)
    c = oracle.ce_shard_combine(parts, mask=mask, z_weight=wz)
    f = oracle.ce_fwd(H, W, y, mask=mask, z_weight=wz)
    logits = torch.from_numpy(H).double() @ torch.from_numpy(W).double().T
    assert np.allclose(c["lse"], torch.logsumexp(logits, 1).numpy(), rtol=1e-14, atol=0)
    assert np.allclose(c["lse"], f["lse"], rtol=1e-14, atol=0)
    assert np.allclose(c["ce"], f["ce"], rtol=1e-13, atol=1e-15)
    assert np.allclose([c["total"], c["ce_mean"], c["z_mean"]], [f["total"], f["ce_mean"], f["z_mean"]],
                       rtol=1e-13)
    dH, dW = oracle.ce_bwd(H, W, y, mask=mask, z_weight=wz, grad_scale=gs)
    dh = np.zeros_like(dH)
    for v0, vs in _shards(V, bounds):
        a, b = oracle.ce_shard_bwd(H, W[v0:v0 + vs], y, v0, V, c["lse"], mask=mask, z_weight=wz,
                                   grad_scale=gs)
        dh += a
        assert np.allclose(b, dW[v0:v0 + vs], rtol=1e-12, atol=1e-16)
    assert np.allclose(dh, dH, rtol=1e-12, atol=1e-16)


def test_shard_contract_refusals():
    H, W, y = _rand(83, 4, 3, 10)
    with pytest.raises(oracle.OracleError) as e:
        oracle.ce_shard_fwd(H, W[:6], y, 5, 10)            # rows 5..10 of a vocabulary of 10
    assert e.value.status == 582
    with pytest.raises(oracle.OracleError) as e:
        oracle.ce_shard_fwd(H, W[:6], np.array([0, 1, 2, 10]), 0, 10)
    assert e.value.status == 586
    # a target held by no shard (the shards leave rows 6..9 out) or by two
    p = oracle.ce_shard_fwd(H, W[:6], y % 6, 0, 10)
    with pytest.raises(oracle.OracleError) as e:
        oracle.ce_shard_combine(np.stack([p, p]))
    assert e.value.status == 586
    y2 = y.copy()
    y2[0] = 8
    p2 = oracle.ce_shard_fwd(H, W[:6], y2, 0, 10)
    with pytest.raises(oracle.OracleError) as e:
        oracle.ce_shard_combine(p2[None])
    assert e.value.status == 586
