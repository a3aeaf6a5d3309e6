"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Tolerances (written here, not derived at run time):
  bf16 inputs, fp32 accumulation: per-token loss and lse |d| <= 2e-3*max(1,|ref|);
                                  gradients relative L2 error <= 1e-2 (whole tensor)
  fp32 inputs:                    per-token loss, lse and scalars |d| <= 1e-6*|ref|
                                  (relative; an absolute 1e-6 only where ref is 0);
                                  gradients relative L2 error <= 1e-5
Where the oracle cannot finish at the full workload size, it computes sampled
tokens (loss, lse, d_hidden rows) and, where affordable, sampled d_weight rows;
the rest is checked through identities that hold at any size.
"""
import math

import numpy as np
import pytest
import torch

import lossk_inputs as li
import oracle

pytestmark = pytest.mark.gpu

class RelTol(float):
    """A loss tolerance applied relative to |ref| alone (the fp32 bound)."""


BF16_LOSS, BF16_GRAD = 2e-3, 1e-2
F32_LOSS, F32_GRAD = RelTol(1e-6), 1e-5


@pytest.fixture(scope="module")
def L():
    from conftest import build_lib
    build_lib()
    import output_projection_cross_gb300 as L
    assert torch.cuda.is_available()
    return L


def _dev(a, dtype):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    if dtype == "bf16":
        return t.to(torch.bfloat16)
    if dtype == "f16":
        return t.to(torch.float16)
    return t


def _tol(dtype):
    """(loss, gradient) tolerances: the 16-bit bound for bf16 and fp16 inputs."""
    return (F32_LOSS, F32_GRAD) if dtype == "fp32" else (BF16_LOSS, BF16_GRAD)


def _redraw(x, dtype, seed, n, d, V, teacher=False):
    """Inputs of another dtype (fp32 / fp16) for a parity case: same recipe."""
    if dtype != "bf16":
        x["hidden"] = li.hidden(seed, n, d, dtype=dtype)
        x["weight"] = li.weight(seed, V, d, dtype=dtype)
        if teacher:
            x["teacher"] = li.teacher(seed, n, V, dtype=dtype)
    return x


def _grad_ref(g, dtype):
    """The gradient a kernel writing `dtype` can return at best.  fp16 outputs
    are compared with the exact gradient rounded to fp16: a softmax gradient
    over a large vocabulary (about 1e-7 per element at 70k entries) lies in
    fp16's subnormal range, whose fixed quantum of 2^-24 no arithmetic can beat;
    bf16 and fp32 keep the exact gradient as the reference."""
    return li.round_to(np.asarray(g, np.float64), "f16").astype(np.float64) if dtype == "f16" else g


def _np(t):
    return t.detach().double().cpu().numpy()


def rel_l2(a, b):
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / nb) if nb > 0 else float(np.linalg.norm(a))


def close_loss(got, ref, tol):
    """|got - ref| <= tol * max(1, |ref|), or, for a RelTol, <= tol * |ref|
    (with tol as an absolute bound only where ref is exactly 0)."""
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    scale = np.where(ref == 0, 1.0, np.abs(ref)) if isinstance(tol, RelTol) else np.maximum(1.0, np.abs(ref))
    err = np.abs(got - ref) / scale
    kind = "relative" if isinstance(tol, RelTol) else "scaled"
    assert err.max() <= tol, f"max {kind} loss error {err.max():.3e} > {float(tol)}"


def _inputs(wl, seed=0, **sizes):
    return li.make(wl, seed=seed, **sizes)


# ---------------------------------------------------------------------------
def test_tiny_fp32_config(L):
    """The fp32 workload at its stated size, full comparison."""
    w = li.WORKLOADS["tiny_fp32_ce"]
    x = _inputs(w)
    H, W, y = _dev(x["hidden"], "fp32"), _dev(x["weight"], "fp32"), _dev(x["targets"], "")
    out = L.lossk_ce_fwd_bwd(H, W, y, chunk=w.chunk)
    torch.cuda.synchronize()
    ref = oracle.ce_fwd(x["hidden"], x["weight"], x["targets"], chunk=w.chunk)
    dH, dW = oracle.ce_bwd(x["hidden"], x["weight"], x["targets"])
    close_loss(_np(out["ce"]), ref["ce"], F32_LOSS)
    close_loss(_np(out["lse"]), ref["lse"], F32_LOSS)
    close_loss(_np(out["scalars"])[:2], [ref["total"], ref["ce_mean"]], F32_LOSS)
    assert rel_l2(_np(out["d_hidden"]), dH) <= F32_GRAD
    assert rel_l2(_np(out["d_weight"]), dW) <= F32_GRAD


SMALL = [  # (n, d, V): several tiles and ragged tails in every dimension
    (1, 64, 8),
    (130, 72, 300),
    (300, 200, 1000),
    (257, 520, 2000),     # 3 d-slices: a cluster of 3
    (128, 256, 512),
    (300, 768, 1000),     # cluster of 3, fewer token tiles than CTAs in the d_weight pass
    (200, 1280, 1500),    # cluster of 5 (one grad slot)
    (130, 2304, 600),     # 9 slices: a cluster of 9 (beyond the portable cluster size)
    (200, 4096, 1000),    # 16 slices: a cluster of 16
    (130, 4352, 600),     # 17 slices: two d-groups of 9
]


@pytest.mark.parametrize("dtype", ["bf16", "fp32", "f16"])
@pytest.mark.parametrize("shape", SMALL)
def test_ce_small_shapes(L, shape, dtype):
    n, d, V = shape
    x = _redraw(_inputs("ce_512x1024x32000", seed=sum(shape), n_tok=n, d_model=d, vocab=V), dtype, 1, n, d, V)
    mask = li.mask(3, n, 0.2) if n > 4 else None
    wz, gs = 1e-3, 0.75
    H, W, y = _dev(x["hidden"], dtype), _dev(x["weight"], dtype), _dev(x["targets"], "")
    m = None if mask is None else _dev(mask, "")
    out = L.lossk_ce_fwd_bwd(H, W, y, loss_mask=m, chunk=min(n, 64), z_weight=wz, grad_scale=gs)
    torch.cuda.synchronize()
    ref = oracle.ce_fwd(x["hidden"], x["weight"], x["targets"], mask=mask, chunk=min(n, 64), z_weight=wz)
    dH, dW = oracle.ce_bwd(x["hidden"], x["weight"], x["targets"], mask=mask, z_weight=wz, grad_scale=gs)
    lt, gt = _tol(dtype)
    close_loss(_np(out["lse"]), ref["lse"], lt)
    close_loss(_np(out["ce"]), ref["ce"], lt)
    close_loss(_np(out["scalars"]), [ref["total"], ref["ce_mean"], ref["z_mean"]], lt)
    assert rel_l2(_np(out["d_hidden"]), dH) <= gt
    assert rel_l2(_np(out["d_weight"]), dW) <= gt


@pytest.mark.parametrize("shape", [(700, 1280, 12000), (300, 1024, 32000)])
def test_ce_persistent_clusters(L, shape):
    """More work units than co-resident clusters, so each backward cluster walks
    several units (slot hand-over across units, accumulator reuse): a cluster of
    5 with one grad slot and ragged splits, and a cluster of 4."""
    n, d, V = shape
    x = _inputs("ce_512x1024x32000", seed=31, n_tok=n, d_model=d, vocab=V)
    mask = li.mask(5, n, 0.1)
    wz, gs = 1e-3, 1.5
    H, W, y = _dev(x["hidden"], "bf16"), _dev(x["weight"], "bf16"), _dev(x["targets"], "")
    out = L.lossk_ce_fwd_bwd(H, W, y, loss_mask=_dev(mask, ""), chunk=64, z_weight=wz, grad_scale=gs)
    torch.cuda.synchronize()
    ref = oracle.ce_fwd(x["hidden"], x["weight"], x["targets"], mask=mask, chunk=64, z_weight=wz)
    dH, dW = oracle.ce_bwd(x["hidden"], x["weight"], x["targets"], mask=mask, z_weight=wz, grad_scale=gs)
    close_loss(_np(out["ce"]), ref["ce"], BF16_LOSS)
    assert rel_l2(_np(out["d_hidden"]), dH) <= BF16_GRAD
    assert rel_l2(_np(out["d_weight"]), dW) <= BF16_GRAD


@pytest.mark.parametrize("direction", ["fkl", "rkl"])
@pytest.mark.parametrize("dtype,shape", [("bf16", (600, 1024, 8192)), ("bf16", (300, 4096, 4096)),
                                         ("f16", (600, 1024, 8192))])
def test_distill_persistent_clusters(L, direction, dtype, shape):
    """Several units per cluster; d_model 4096 runs one cluster of 16 CTAs."""
    n, d, V = shape
    x = _inputs("distill_z_4096x2048", seed=32, n_tok=n, d_model=d, vocab=V)
    x = _redraw(x, dtype, 3, n, d, V, teacher=True)
    mask = li.mask(6, n, 0.1)
    out = L.lossk_distill_fwd_bwd(_dev(x["hidden"], dtype), _dev(x["weight"], dtype),
                                  _dev(x["teacher"], dtype), direction, temperature=2.0,
                                  loss_mask=_dev(mask, ""), z_weight=1e-3)
    torch.cuda.synchronize()
    r = oracle.distill(x["hidden"], x["weight"], x["teacher"], direction, temperature=2.0,
                       mask=mask, z_weight=1e-3)
    close_loss(_np(out["per_token"]), r["per_token"], BF16_LOSS)
    assert rel_l2(_np(out["d_hidden"]), r["dH"]) <= BF16_GRAD
    assert rel_l2(_np(out["d_weight"]), r["dW"]) <= BF16_GRAD


def test_ce_fwd_and_bwd_entry_points_agree_with_fused(L):
    """The separate calls run the forward statistics and both backward passes;
    the training-step call folds d_hidden into its forward pass (a per-token
    reference shift instead of the lse).  Same quantities, different rounding:
    they agree far inside the oracle tolerances, and the separate calls are
    bit-stable."""
    n, d, V = 200, 128, 1500
    x = _inputs("ce_512x1024x32000", seed=5, n_tok=n, d_model=d, vocab=V)
    H, W, y = _dev(x["hidden"], "bf16"), _dev(x["weight"], "bf16"), _dev(x["targets"], "")
    f = L.lossk_ce_fwd(H, W, y, chunk=32, z_weight=0.01)
    b = L.lossk_ce_bwd(H, W, y, f["lse"], z_weight=0.01, grad_scale=2.0)
    fb = L.lossk_ce_fwd_bwd(H, W, y, chunk=32, z_weight=0.01, grad_scale=2.0)
    f2 = L.lossk_ce_fwd(H, W, y, chunk=32, z_weight=0.01)
    torch.cuda.synchronize()
    assert torch.equal(f["lse"], f2["lse"]) and torch.equal(f["scalars"], f2["scalars"])
    close_loss(_np(fb["lse"]), _np(f["lse"]), 1e-5)
    close_loss(_np(fb["scalars"]), _np(f["scalars"]), 1e-5)
    assert rel_l2(_np(fb["d_hidden"]), _np(b["d_hidden"])) <= 4e-3
    assert rel_l2(_np(fb["d_weight"]), _np(b["d_weight"])) <= 1e-4
    # either gradient may be skipped
    only_w = L.lossk_ce_bwd(H, W, y, f["lse"], z_weight=0.01, grad_scale=2.0, want_d_hidden=False)
    torch.cuda.synchronize()
    assert only_w["d_hidden"] is None and torch.equal(only_w["d_weight"], b["d_weight"])


def _kernels_run(L, fn):
    L.lossk_profile_enable(True)
    L.lossk_profile_read(reset=True)
    fn()
    torch.cuda.synchronize()
    k = L.lossk_profile_read(reset=True)
    L.lossk_profile_enable(False)
    return k


def test_fused_forward_dhidden_path_is_the_one_that_runs(L):
    n, d, V = 300, 256, 2000
    x = _inputs("ce_512x1024x32000", seed=8, n_tok=n, d_model=d, vocab=V)
    H, W, y = _dev(x["hidden"], "bf16"), _dev(x["weight"], "bf16"), _dev(x["targets"], "")
    k = _kernels_run(L, lambda: L.lossk_ce_fwd_bwd(H, W, y, z_weight=1e-3))
    assert {"validate", "tc_fused", "merge_fused", "combine_dh", "tc_cols"} <= set(k)
    # the target logits come with the validation launch on this path
    assert "tc_stats" not in k and "tc_rows" not in k and "tgt_logit" not in k
    # without d_hidden there is nothing to fold: the separate forward runs
    k = _kernels_run(L, lambda: L.lossk_ce_fwd_bwd(H, W, y, want_d_hidden=False))
    assert "tc_stats" in k and "tc_fused" not in k


def test_fused_path_recomputes_rows_beyond_its_shift(L):
    """Token 7's target logit sits 160 nats under its row maximum: the fused
    pass's shifted terms overflow for that row, the call notices and
    recomputes every output on the separate passes, which match the oracle."""
    n, d, V = 130, 64, 1000
    x = _inputs("ce_512x1024x32000", seed=9, n_tok=n, d_model=d, vocab=V)
    Hn, Wn, yn = x["hidden"].copy(), x["weight"].copy(), x["targets"].copy()
    Hn[7, :] = 1.0
    Wn[3, :] = 2.5          # s[7][3] = 64 * 2.5 = 160
    Wn[5, :] = 0.0          # s[7][5] = 0
    yn[7] = 5
    Hn, Wn = li.to_bf16_values(Hn), li.to_bf16_values(Wn)
    H, W, y = _dev(Hn, "bf16"), _dev(Wn, "bf16"), _dev(yn, "")
    box = {}
    k = _kernels_run(L, lambda: box.update(o=L.lossk_ce_fwd_bwd(H, W, y, z_weight=1e-4, grad_scale=1.0)))
    assert "tc_fused" in k and "tc_stats" in k and "tc_rows" in k
    o = box["o"]
    ref = oracle.ce_fwd(Hn, Wn, yn, z_weight=1e-4)
    dH, dW = oracle.ce_bwd(Hn, Wn, yn, z_weight=1e-4, grad_scale=1.0)
    assert abs(ref["ce"][7] - 160.0) < 1.0
    close_loss(_np(o["ce"]), ref["ce"], BF16_LOSS)
    close_loss(_np(o["lse"]), ref["lse"], BF16_LOSS)
    assert rel_l2(_np(o["d_hidden"]), dH) <= BF16_GRAD
    assert rel_l2(_np(o["d_weight"]), dW) <= BF16_GRAD


def test_config_512x1024x32000_full(L):
    w = li.WORKLOADS["ce_512x1024x32000"]
    x = _inputs(w)
    H, W, y = _dev(x["hidden"], "bf16"), _dev(x["weight"], "bf16"), _dev(x["targets"], "")
    out = L.lossk_ce_fwd_bwd(H, W, y, chunk=w.chunk)
    torch.cuda.synchronize()
    ref = oracle.ce_fwd(x["hidden"], x["weight"], x["targets"], chunk=w.chunk)
    dH, dW = oracle.ce_bwd(x["hidden"], x["weight"], x["targets"])
    close_loss(_np(out["ce"]), ref["ce"], BF16_LOSS)
    close_loss(_np(out["lse"]), ref["lse"], BF16_LOSS)
    close_loss(_np(out["scalars"])[:2], [ref["total"], ref["ce_mean"]], BF16_LOSS)
    assert rel_l2(_np(out["d_hidden"]), dH) <= BF16_GRAD
    assert rel_l2(_np(out["d_weight"]), dW) <= BF16_GRAD


_QWEN3_ORACLE = {}


def _qwen3_oracle(x, w):
    """The oracle's full forward at the Qwen3 head shape (bf16 inputs), computed once."""
    if not _QWEN3_ORACLE:
        _QWEN3_ORACLE.update(oracle.ce_fwd(x["hidden"], x["weight"], x["targets"], chunk=w.chunk))
    return _QWEN3_ORACLE


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_qwen3_head_full_size_sampled(L, dtype):
    """n=2048, d=1024, V=151936, Zipf targets: the launch configuration the bench
    times (bf16: the training step's single-pass forward + d_hidden; fp16: the
    separate passes with the grad tiles' common factor applied at the store)."""
    w = li.WORKLOADS["qwen3_0p6b_head"]
    x = _redraw(_inputs(w), dtype, 0, w.n_tok, w.d_model, w.vocab)
    H, W, y = _dev(x["hidden"], dtype), _dev(x["weight"], dtype), _dev(x["targets"], "")
    out = L.lossk_ce_fwd_bwd(H, W, y, chunk=w.chunk)
    torch.cuda.synchronize()
    rows = np.random.default_rng(7).choice(w.n_tok, 48, replace=False)
    rows.sort()
    s = oracle.ce_token_rows(x["hidden"], x["weight"], x["targets"], rows)
    close_loss(_np(out["lse"])[rows], s["lse"], BF16_LOSS)
    close_loss(_np(out["ce"])[rows], s["lse"] - s["tgt"], BF16_LOSS)
    assert rel_l2(_np(out["d_hidden"])[rows], s["dH"]) <= BF16_GRAD
    # d_weight rows: the oracle needs every token's lse
    full = _qwen3_oracle(x, w) if dtype == "bf16" else oracle.ce_fwd(x["hidden"], x["weight"], x["targets"],
                                                                      chunk=w.chunk)
    close_loss(_np(out["lse"]), full["lse"], BF16_LOSS)
    close_loss(_np(out["scalars"])[:1], [full["total"]], BF16_LOSS)
    vrows = np.concatenate([np.unique(x["targets"])[:24],
                            np.random.default_rng(8).choice(w.vocab, 24, replace=False)])
    dw = oracle.ce_dweight_rows(x["hidden"], x["weight"], x["targets"], full["lse"], vrows)
    assert rel_l2(_np(out["d_weight"])[vrows], dw) <= BF16_GRAD
    # any-size identity: d_weight summed over the vocabulary cancels (no z-loss)
    dws = out["d_weight"].double().sum(0).cpu().numpy()
    assert np.abs(dws).max() <= 1e-2 * np.abs(_np(out["d_weight"])).max()


def test_largest_vocab(L):
    """The largest vocabulary the contract accepts (2^24) at the largest chunk
    it then allows (chunk * vocab = 2^27), with a few tokens: 65536 vocabulary
    supertiles per token tile, 2 GB of bf16 weight and a 4.3 GB fp32 d_weight.
    Every token's loss and d_hidden row and sampled d_weight rows against the
    oracle, plus the vocabulary-sum identity of d_weight."""
    n, d, V = 8, 64, 1 << 24
    g = torch.Generator(device="cuda").manual_seed(11)
    H = torch.randn(n, d, device="cuda", generator=g).to(torch.bfloat16)
    W = (torch.randn(V, d, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    y = torch.randint(0, V, (n,), device="cuda", generator=g)
    y[0], y[1] = 0, V - 1                       # the first and the last vocabulary row
    out = L.lossk_ce_fwd_bwd(H, W, y, chunk=8)
    torch.cuda.synchronize()
    Hn, Wn, yn = H.float().cpu().numpy(), W.float().cpu().numpy(), y.cpu().numpy()
    s = oracle.ce_token_rows(Hn, Wn, yn, np.arange(n))
    close_loss(_np(out["lse"]), s["lse"], BF16_LOSS)
    close_loss(_np(out["ce"]), s["lse"] - s["tgt"], BF16_LOSS)
    assert rel_l2(_np(out["d_hidden"]), s["dH"]) <= BF16_GRAD
    vrows = np.concatenate([np.unique(yn), np.random.default_rng(12).choice(V, 24, replace=False)])
    dw = oracle.ce_dweight_rows(Hn, Wn, yn, s["lse"], vrows)
    assert rel_l2(_np(out["d_weight"][torch.from_numpy(vrows).cuda()]), dw) <= BF16_GRAD
    dws = out["d_weight"].double().sum(0).cpu().numpy()
    assert np.abs(dws).max() <= 1e-2 * np.abs(_np(out["d_weight"][torch.from_numpy(vrows).cuda()])).max()


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_d_weight_many_token_supertiles(L, dtype):
    """1500 tokens at d_model 128: clusters of one CTA, each owning all six token
    supertiles of a unit, more than the d_weight epilogue keeps in its shared
    parameter copy; it then loads the parameters tile by tile.  Label CE and
    distillation (the TMA teacher-block variant of the pass)."""
    n, d, V = 1500, 128, 2000
    x = _redraw(_inputs("ce_512x1024x32000", seed=71, n_tok=n, d_model=d, vocab=V), dtype, 3, n, d, V)
    mask = li.mask(4, n, 0.1)
    H, W, y = _dev(x["hidden"], dtype), _dev(x["weight"], dtype), _dev(x["targets"], "")
    out = L.lossk_ce_fwd_bwd(H, W, y, loss_mask=_dev(mask, ""), z_weight=1e-3, grad_scale=0.5)
    torch.cuda.synchronize()
    dH, dW = oracle.ce_bwd(x["hidden"], x["weight"], x["targets"], mask=mask, z_weight=1e-3, grad_scale=0.5)
    lt, gt = _tol(dtype)
    assert rel_l2(_np(out["d_hidden"]), dH) <= gt
    assert rel_l2(_np(out["d_weight"]), dW) <= gt
    Tt = li.round_to((np.random.default_rng(72).standard_normal((n, V)) * 3).astype(np.float32), dtype)
    o = L.lossk_distill_fwd_bwd(H, W, _dev(Tt, dtype), "rkl", temperature=2.0, loss_mask=_dev(mask, ""),
                                z_weight=1e-3, grad_scale=0.5)
    torch.cuda.synchronize()
    r = oracle.distill(x["hidden"], x["weight"], Tt, "rkl", temperature=2.0, mask=mask, z_weight=1e-3,
                       grad_scale=0.5)
    close_loss(_np(o["per_token"]), r["per_token"], lt)
    assert rel_l2(_np(o["d_hidden"]), r["dH"]) <= gt
    assert rel_l2(_np(o["d_weight"]), r["dW"]) <= gt


def test_ce_z_mask_reduced_full(L):
    """The CE + z-loss + mask recipe at a size the oracle finishes in seconds."""
    w = li.WORKLOADS["ce_z_8192x4096x128256"]
    x = _inputs(w, n_tok=640, d_model=512, vocab=5000)
    mask = li.mask(0, 640, w.mask_frac)
    H, W, y = _dev(x["hidden"], "bf16"), _dev(x["weight"], "bf16"), _dev(x["targets"], "")
    out = L.lossk_ce_fwd_bwd(H, W, y, loss_mask=_dev(mask, ""), chunk=128, z_weight=w.z_weight)
    torch.cuda.synchronize()
    ref = oracle.ce_fwd(x["hidden"], x["weight"], x["targets"], mask=mask, chunk=128, z_weight=w.z_weight)
    dH, dW = oracle.ce_bwd(x["hidden"], x["weight"], x["targets"], mask=mask, z_weight=w.z_weight)
    close_loss(_np(out["ce"]), ref["ce"], BF16_LOSS)
    close_loss(_np(out["scalars"]), [ref["total"], ref["ce_mean"], ref["z_mean"]], BF16_LOSS)
    assert rel_l2(_np(out["d_hidden"]), dH) <= BF16_GRAD
    assert rel_l2(_np(out["d_weight"]), dW) <= BF16_GRAD


def test_ce_z_mask_full_size_sampled(L):
    """n=8192, d=4096, V=128256, z weight 1e-4, 5% masked: sampled tokens + identities."""
    w = li.WORKLOADS["ce_z_8192x4096x128256"]
    x = _inputs(w)
    mask = x["mask"]
    H, W, y = _dev(x["hidden"], "bf16"), _dev(x["weight"], "bf16"), _dev(x["targets"], "")
    out = L.lossk_ce_fwd_bwd(H, W, y, loss_mask=_dev(mask, ""), chunk=w.chunk, z_weight=w.z_weight)
    torch.cuda.synchronize()
    masked = np.flatnonzero(mask == 0)[:4]
    rows = np.sort(np.concatenate([np.random.default_rng(9).choice(w.n_tok, 20, replace=False), masked]))
    s = oracle.ce_token_rows(x["hidden"], x["weight"], x["targets"], rows, mask=mask, z_weight=w.z_weight)
    close_loss(_np(out["lse"])[rows], s["lse"], BF16_LOSS)
    ce_ref = np.where(mask[rows] != 0, s["lse"] - s["tgt"], 0.0)
    close_loss(_np(out["ce"])[rows], ce_ref, BF16_LOSS)
    assert rel_l2(_np(out["d_hidden"])[rows], s["dH"]) <= BF16_GRAD
    assert np.all(_np(out["d_hidden"])[masked] == 0)
    # identity: sum_v G_tv = alpha_t * 2 wz lse_t, so sum_v dW_v = sum_t alpha_t 2 wz lse_t H_t,
    # up to the bf16 rounding of each G element (unit roundoff 2^-8): sum_v |dG_tv| <=
    # 2^-8 * sum_v |G_tv| <= 2^-8 * alpha_t (2 + 2 wz lse_t), which bounds each column k
    # by sum_t |H_tk| times that.
    lse = out["lse"].double()
    m = torch.from_numpy(mask).cuda().double()
    alpha = m / m.sum()
    expect = ((alpha * 2 * w.z_weight * lse)[:, None] * H.double()).sum(0)
    bound = ((alpha * 2.0 ** -8 * (2 + 2 * w.z_weight * lse))[:, None] * H.double().abs()).sum(0)
    got = out["d_weight"].double().sum(0)
    assert bool(((got - expect).abs() <= bound * 1.05 + 1e-9).all())
    # every token and the reduced scalars against the oracle's full-size values
    # (tests/golden/make_full_size_goldens.py, computed with the oracle alone)
    g = _full_size_golden("ce_z_8192x4096x128256", x)
    close_loss(_np(out["lse"]), g["lse"], BF16_LOSS)
    close_loss(_np(out["ce"]), g["ce"], BF16_LOSS)
    close_loss(_np(out["scalars"]), g["scalars"], BF16_LOSS)
    vrows = torch.from_numpy(g["vrows"]).cuda()
    assert rel_l2(_np(out["d_weight"][vrows]), g["dweight_rows"].astype(np.float64)) <= BF16_GRAD


# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["bf16", "fp32", "f16"])
@pytest.mark.parametrize("direction", ["ce", "fkl", "rkl"])
@pytest.mark.parametrize("T", [1.0, 2.0])
def test_distill_small(L, dtype, direction, T):
    n, d, V = 200, 136, 1032
    x = _inputs("distill_z_4096x2048", seed=11, n_tok=n, d_model=d, vocab=V)
    if dtype == "fp32":
        x["hidden"] = li.hidden(2, n, d, dtype="fp32")
        x["weight"] = li.weight(2, V, d, dtype="fp32")
    if dtype == "f16":
        x = _redraw(x, "f16", 2, n, d, V, teacher=True)
    mask = li.mask(1, n, 0.1)
    wz, gs = 1e-3, 1.25
    Tt = x["teacher"]
    H, W = _dev(x["hidden"], dtype), _dev(x["weight"], dtype)
    teach = _dev(Tt, dtype)
    out = L.lossk_distill_fwd_bwd(H, W, teach, direction, temperature=T, loss_mask=_dev(mask, ""),
                                  chunk=50, z_weight=wz, grad_scale=gs)
    torch.cuda.synchronize()
    r = oracle.distill(x["hidden"], x["weight"], Tt, direction, temperature=T, mask=mask, chunk=50,
                       z_weight=wz, grad_scale=gs)
    lt, gt = _tol(dtype)
    close_loss(_np(out["per_token"]), r["per_token"], lt)
    close_loss(_np(out["lse"]), r["lse"], lt)
    close_loss(_np(out["scalars"]), [r["total"], r["distill_mean"], r["z_mean"]], lt)
    assert rel_l2(_np(out["d_hidden"]), r["dH"]) <= gt
    assert rel_l2(_np(out["d_weight"]), r["dW"]) <= gt


@pytest.mark.parametrize("direction", ["fkl", "rkl", "ce"])
def test_distill_full_size_sampled(L, direction):
    """n=4096, d=2048, V=151936, teacher N(0,3) bf16, T=2, 10% masked, z 1e-4."""
    w = li.WORKLOADS["distill_z_4096x2048"]
    x = _cached_distill()
    mask = x["mask"]
    H, W, teach = x["H"], x["W"], x["T"]
    out = L.lossk_distill_fwd_bwd(H, W, teach, direction, temperature=w.temperature,
                                  loss_mask=x["m"], chunk=w.chunk, z_weight=w.z_weight)
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(12).choice(w.n_tok, 12, replace=False))
    s = oracle.distill_token_rows(x["hidden"], x["weight"], x["teacher"], direction, rows,
                                  temperature=w.temperature, mask=mask, z_weight=w.z_weight)
    per = np.where(mask[rows] != 0, s["loss"], 0.0)
    close_loss(_np(out["per_token"])[rows], per, BF16_LOSS)
    close_loss(_np(out["lse"])[rows], s["lse"], BF16_LOSS)
    assert rel_l2(_np(out["d_hidden"])[rows], s["dH"]) <= BF16_GRAD
    # identity: every objective's gradient row sums to alpha_t/T * 2 wz lse_t (q and p
    # both sum to one; for reverse-KL the q-weighted log-ratio sums to L_t), up to the
    # bf16 rounding of G (unit roundoff 2^-8): sum_v |dG_tv| <= 2^-8 alpha_t/T (sum_v q
    # (1 + 2 wz lse) + p [+ q |log q - log p - L| for reverse-KL]) <= 2^-8 * 8 alpha_t/T.
    lse = out["lse"].double()
    m = x["m"].double()
    alpha = m / m.sum()
    T = w.temperature
    expect = ((alpha * 2 * w.z_weight * lse / T)[:, None] * H.double()).sum(0)
    got = out["d_weight"].double().sum(0)
    bound = ((alpha * 8 * 2.0 ** -8 / T)[:, None] * H.double().abs()).sum(0)
    err = (got - expect).abs()
    assert bool((err <= bound).all()), float((err / bound).max())
    # and the signal is resolved: the relative L2 error of the row sum is small
    assert float(torch.linalg.norm(got - expect) / torch.linalg.norm(expect)) <= 5e-2
    # every token, the reduced scalars and sampled d_weight rows against the
    # oracle's full-size values (tests/golden/make_full_size_goldens.py)
    gd = _full_size_golden("distill_z_4096x2048", {k: x[k] for k in ("hidden", "weight", "targets", "mask",
                                                                      "teacher")})
    per = np.where(mask != 0, gd[f"{direction}_loss"], 0.0)
    close_loss(_np(out["per_token"]), per, BF16_LOSS)
    close_loss(_np(out["lse"]), gd[f"{direction}_lse"], BF16_LOSS)
    close_loss(_np(out["scalars"]), gd[f"{direction}_scalars"], BF16_LOSS)
    vrows = torch.from_numpy(gd["vrows"]).cuda()
    assert rel_l2(_np(out["d_weight"][vrows]), gd[f"{direction}_dweight_rows"].astype(np.float64)) <= BF16_GRAD


_DISTILL_CACHE = {}


def _full_size_golden(name, x):
    """The oracle's stored values for a full-size workload, after checking that
    this machine drew the same inputs (the stored SHA-256 fingerprint)."""
    import importlib.util
    import os
    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    spec = importlib.util.spec_from_file_location("make_full_size_goldens",
                                                  os.path.join(here, "make_full_size_goldens.py"))
    mk = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mk)
    g = dict(np.load(mk.golden_path(name)))
    assert str(g["fingerprint"]) == mk.fingerprint(x), "the seeded inputs differ from the stored oracle values'"
    return g


def _cached_distill():
    if not _DISTILL_CACHE:
        w = li.WORKLOADS["distill_z_4096x2048"]
        x = _inputs(w)
        _DISTILL_CACHE.update(x)
        _DISTILL_CACHE["H"] = _dev(x["hidden"], "bf16")
        _DISTILL_CACHE["W"] = _dev(x["weight"], "bf16")
        _DISTILL_CACHE["T"] = _dev(x["teacher"], "bf16")
        _DISTILL_CACHE["m"] = _dev(x["mask"], "")
    return _DISTILL_CACHE


# ---------------------------------------------------------------------------
# V 9 and 4099: rows that are not 16-byte multiples (the element-wise loops);
# 1000: fewer 16-byte vectors than threads; 70008 and 151936: several rounds of
# four vectors per thread, the last one ragged
@pytest.mark.parametrize("dtype", ["bf16", "fp32", "f16"])
@pytest.mark.parametrize("V", [9, 1000, 4099, 70008, 151936])
def test_from_logits(L, dtype, V):
    n = 37 if V > 10000 else 129
    g = np.random.default_rng(V)
    X = li.round_to((g.standard_normal((n, V)) * 2).astype(np.float32), dtype)
    y = g.integers(0, V, n).astype(np.int64)
    mask = (np.arange(n) % 7 != 3).astype(np.uint8)
    wz, gs = 1e-2, 1.5
    out = L.lossk_ce_from_logits(_dev(X, dtype), _dev(y, ""), loss_mask=_dev(mask, ""), z_weight=wz,
                                 grad_scale=gs, want_grad=True)
    torch.cuda.synchronize()
    r = oracle.ce_from_logits(X, y, mask=mask, z_weight=wz, grad_scale=gs, want_grad=True)
    lt, gt = _tol(dtype)
    close_loss(_np(out["lse"]), r["lse"], lt)
    close_loss(_np(out["ce"]), r["ce"], lt)
    close_loss(_np(out["scalars"]), [r["total"], r["ce_mean"], r["z_mean"]], lt)
    assert rel_l2(_np(out["grad_logits"]), _grad_ref(r["grad"], dtype)) <= gt


def test_logits_rows_full_size_sampled(L):
    """The launch configuration the bench times for the two losses over given
    logits: 2048 rows of 151936 bf16 logits, with the gradient.  Sampled rows
    against the oracle (with the gradient scale rescaled so that the sample's
    token mean weights its rows as the full batch's does)."""
    n, V = 2048, 151936
    g = torch.Generator(device="cuda").manual_seed(5)
    X = torch.randn(n, V, device="cuda", generator=g).to(torch.bfloat16)
    T = (torch.randn(n, V, device="cuda", generator=g) * 3).to(torch.bfloat16)
    y = torch.randint(0, V, (n,), device="cuda", generator=g)
    rows = np.array([0, 1, 777, 1024, 1500, n - 1])
    gs = 1.5
    out = L.lossk_ce_from_logits(X, y, z_weight=1e-4, grad_scale=gs, want_grad=True)
    torch.cuda.synchronize()
    Xs, ys = _np(X[rows]), y[rows].cpu().numpy()
    r = oracle.ce_from_logits(Xs, ys, z_weight=1e-4, grad_scale=gs * len(rows) / n, want_grad=True)
    lt, gt = _tol("bf16")
    close_loss(_np(out["lse"])[rows], r["lse"], lt)
    close_loss(_np(out["ce"])[rows], r["ce"], lt)
    assert rel_l2(_np(out["grad_logits"][rows]), r["grad"]) <= gt
    del out
    for direction in ("fkl", "rkl"):
        o = L.lossk_distill_from_logits(X, T, direction, temperature=2.0, z_weight=1e-4, grad_scale=gs,
                                        want_grad=True)
        torch.cuda.synchronize()
        r = oracle.distill_from_logits(Xs, _np(T[rows]), direction, temperature=2.0, z_weight=1e-4,
                                       grad_scale=gs * len(rows) / n)
        close_loss(_np(o["per_token"])[rows], r["per_token"], lt)
        close_loss(_np(o["lse"])[rows], r["lse"], lt)
        assert rel_l2(_np(o["grad_logits"][rows]), r["grad"]) <= gt
        del o


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("V", [1000, 1003])
def test_from_logits_masked_vocabulary(L, dtype, V):
    """-inf logits (vocabulary entries masked out of a row) have probability 0:
    finite lse and ce, a zero gradient there.  Whole 16-byte vectors of -inf
    (V 1000) and the element-wise path (V 1003); one row keeps a single finite
    entry, its target."""
    n = 40
    g = np.random.default_rng(V + 3)
    X = li.round_to((g.standard_normal((n, V)) * 2).astype(np.float32), dtype)
    X[:, 8:600] = -np.inf
    X[:, : 3] = -np.inf
    X[5, :] = -np.inf
    y = g.integers(600, V, n).astype(np.int64)
    X[5, y[5]] = 1.25
    out = L.lossk_ce_from_logits(_dev(X, dtype), _dev(y, ""), z_weight=1e-3, want_grad=True)
    torch.cuda.synchronize()
    r = oracle.ce_from_logits(X, y, z_weight=1e-3, want_grad=True)
    assert np.isfinite(_np(out["lse"])).all() and np.isfinite(_np(out["grad_logits"])).all()
    lt, gt = _tol(dtype)
    close_loss(_np(out["lse"]), r["lse"], lt)
    close_loss(_np(out["ce"]), r["ce"], lt)
    assert rel_l2(_np(out["grad_logits"]), r["grad"]) <= gt
    assert np.all(_np(out["grad_logits"])[:, 8:600] == 0)


def test_from_logits_uniform_golden(L):
    """6 tokens, vocab 9, every logit 0.25 -> mean loss ln 9 (the pages' worked example)."""
    X = torch.full((6, 9), 0.25, device="cuda", dtype=torch.float32)
    y = torch.tensor([0, 3, 6, 0, 3, 6], device="cuda")
    out = L.lossk_ce_from_logits(X, y)
    torch.cuda.synchronize()
    assert abs(out["scalars"][0].item() - 2.1972245773362196) <= 1e-6 * 2.1972245773362196


# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_chunk_invariance_and_determinism(L, dtype):
    n, d, V = 300, 128, 3000
    x = _inputs("ce_512x1024x32000", seed=21, n_tok=n, d_model=d, vocab=V)
    H, W, y = _dev(x["hidden"], dtype), _dev(x["weight"], dtype), _dev(x["targets"], "")
    if dtype == "fp32":
        H, W = H.float(), W.float()
    base = L.lossk_ce_fwd_bwd(H, W, y, chunk=n, z_weight=0.01)
    for chunk in (1, 7, 64, 256):
        o = L.lossk_ce_fwd_bwd(H, W, y, chunk=chunk, z_weight=0.01)
        torch.cuda.synchronize()
        for k in ("lse", "ce", "scalars", "d_hidden", "d_weight"):
            assert torch.equal(o[k], base[k]), (chunk, k)


def test_calls_on_two_streams_match_one_stream(L):
    """Training-step calls from two host threads, each on its own stream and
    workspace (each caller stream gets its own helper stream for the token mean
    and d_hidden's combine), give the bits of the same calls made one at a
    time."""
    import threading

    n, d, V = 512, 256, 4000
    x = _inputs("ce_512x1024x32000", seed=31, n_tok=n, d_model=d, vocab=V)
    H, W, y = _dev(x["hidden"], "bf16"), _dev(x["weight"], "bf16"), _dev(x["targets"], "")
    H2 = (H.float() * 0.5).to(torch.bfloat16)
    ref = [L.lossk_ce_fwd_bwd(H, W, y, z_weight=0.01), L.lossk_ce_fwd_bwd(H2, W, y, z_weight=0.01)]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for _ in range(3):
        out = [None, None]

        def run(i, Hx):
            with torch.cuda.stream(streams[i]):
                out[i] = L.lossk_ce_fwd_bwd(Hx, W, y, z_weight=0.01, stream=streams[i])

        th = [threading.Thread(target=run, args=(0, H)), threading.Thread(target=run, args=(1, H2))]
        for t in th:
            t.start()
        for t in th:
            t.join()
        torch.cuda.synchronize()
        for i in range(2):
            for k in ("lse", "ce", "scalars", "d_hidden", "d_weight"):
                assert torch.equal(out[i][k], ref[i][k]), (i, k)


def test_zero_weight_closed_form(L):
    n, d, V = 100, 64, 1000
    H = torch.randn(n, d, device="cuda").to(torch.bfloat16)
    W = torch.zeros(V, d, device="cuda", dtype=torch.bfloat16)
    y = torch.randint(0, V, (n,), device="cuda")
    o = L.lossk_ce_fwd_bwd(H, W, y, z_weight=0.5)
    torch.cuda.synchronize()
    lv = math.log(V)
    assert torch.allclose(o["lse"].double(), torch.full((n,), lv, dtype=torch.float64, device="cuda"), atol=1e-5)
    s = o["scalars"].cpu().numpy()
    assert abs(s[1] - lv) <= 1e-5 and abs(s[2] - lv * lv) <= 1e-4


def test_z_weight_zero_path_is_bit_identical_to_no_z(L):
    """z gated off: the loss equals its ce mean exactly and gradients equal a
    second call's bits."""
    n, d, V = 150, 64, 700
    x = _inputs("ce_512x1024x32000", seed=2, n_tok=n, d_model=d, vocab=V)
    H, W, y = _dev(x["hidden"], "bf16"), _dev(x["weight"], "bf16"), _dev(x["targets"], "")
    a = L.lossk_ce_fwd_bwd(H, W, y, z_weight=0.0)
    torch.cuda.synchronize()
    assert a["scalars"][0].item() == a["scalars"][1].item()


def test_refusals_leave_outputs_untouched(L):
    n, d, V = 64, 64, 500
    H = torch.randn(n, d, device="cuda").to(torch.bfloat16)
    W = torch.randn(V, d, device="cuda").to(torch.bfloat16)
    for bad in (-1, V):
        y = torch.randint(0, V, (n,), device="cuda")
        y[5] = bad
        lse = torch.full((n,), 7.0, device="cuda")
        with pytest.raises(L.LosskError) as e:
            L.lossk_ce_fwd(H, W, y, lse_out=lse)
        assert e.value.status == 586
        assert torch.all(lse == 7.0)
    y = torch.randint(0, V, (n,), device="cuda")
    assert L.lossk_targets_check(y, V) == 580
    y[0] = V
    assert L.lossk_targets_check(y, V) == 586
    with pytest.raises(L.LosskError) as e:
        L.lossk_ce_fwd(H, W, torch.randint(0, V, (n,), device="cuda"), chunk=(1 << 27) // V + 1)
    assert e.value.status == 587
    V8 = 512          # a teacher row pitch of 16-byte multiples, so 591 does not fire first
    W8 = torch.randn(V8, d, device="cuda").to(torch.bfloat16)
    with pytest.raises(L.LosskError) as e:
        L.lossk_distill_fwd_bwd(H, W8, torch.zeros(n, V8, device="cuda", dtype=torch.bfloat16), 5)
    assert e.value.status == 588
    with pytest.raises(L.LosskError) as e:    # vocab 500: bf16 teacher rows are not 16-byte multiples
        L.lossk_distill_fwd_bwd(H, W, torch.zeros(n, V, device="cuda", dtype=torch.bfloat16), 0)
    assert e.value.status == 591


@pytest.mark.parametrize("V", [500, 1000, 151936])
def test_from_logits_refusal_touches_no_output(L, V):
    """Cross-entropy from logits refuses a target out of range before its
    kernels run: no output changes, with or without a gradient (V 1000 and 151936:
    16-byte vector loops; 500: rows that are not 16-byte multiples)."""
    n = 40
    X = torch.randn(n, V, device="cuda").to(torch.bfloat16)
    for want in (False, True):
        for bad in (-2, V):
            y = torch.randint(0, V, (n,), device="cuda")
            y[n - 3] = bad
            lse = torch.full((n,), 7.0, device="cuda")
            ce = torch.full((n,), 8.0, device="cuda")
            sc = torch.full((3,), 9.0, dtype=torch.float64, device="cuda")
            gl = torch.full((n, V), 1.5, device="cuda", dtype=torch.bfloat16)
            with pytest.raises(L.LosskError) as e:
                L.lossk_ce_from_logits(X, y, lse_out=lse, ce_out=ce, scalars_out=sc,
                                       grad_logits=gl if want else None, want_grad=want)
            assert e.value.status == 586
            torch.cuda.synchronize()
            assert torch.all(lse == 7.0) and torch.all(ce == 8.0) and torch.all(sc == 9.0)
            assert torch.all(gl == 1.5)
    y = torch.randint(0, V, (n,), device="cuda")
    out = L.lossk_ce_from_logits(X, y, want_grad=True)
    torch.cuda.synchronize()
    r = oracle.ce_from_logits(_np(X), y.cpu().numpy(), want_grad=True)
    close_loss(_np(out["lse"]), r["lse"], _tol("bf16")[0])
    assert rel_l2(_np(out["grad_logits"]), r["grad"]) <= _tol("bf16")[1]


@pytest.mark.parametrize("shape", [(64, 64, 500), (300, 256, 4000)])
def test_training_step_refusal_touches_no_output(L, shape):
    """The bf16 training step validates without waiting: its later kernels
    return at once on the device when a target is out of range.  Every output
    (including d_hidden, which the fused pass writes directly when there is a
    single vocabulary split, as at the first shape) must keep its contents, with
    and without accumulation; a valid call on the same workspace then works."""
    n, d, V = shape
    H = torch.randn(n, d, device="cuda").to(torch.bfloat16)
    W = (torch.randn(V, d, device="cuda") * 0.05).to(torch.bfloat16)
    ws = L.workspace(L.lossk.KIND_CE_FWD_BWD, n, d, V, L.lossk.BF16)
    for flags in (0, L.lossk.ACCUMULATE_GRADS):
        for bad in (-3, V):
            y = torch.randint(0, V, (n,), device="cuda")
            y[n // 2] = bad
            outs = dict(lse_out=torch.full((n,), 7.0, device="cuda"), ce_out=torch.full((n,), 8.0, device="cuda"),
                        scalars_out=torch.full((3,), 9.0, dtype=torch.float64, device="cuda"),
                        d_hidden=torch.full((n, d), 1.5, device="cuda"), d_weight=torch.full((V, d), 2.5, device="cuda"))
            with pytest.raises(L.LosskError) as e:
                L.lossk_ce_fwd_bwd_ex(H, W, y, flags=flags, z_weight=1e-3, ws=ws, **outs)
            assert e.value.status == 586
            torch.cuda.synchronize()
            assert torch.all(outs["lse_out"] == 7.0) and torch.all(outs["ce_out"] == 8.0)
            assert torch.all(outs["scalars_out"] == 9.0)
            assert torch.all(outs["d_hidden"] == 1.5) and torch.all(outs["d_weight"] == 2.5)
    y = torch.randint(0, V, (n,), device="cuda")
    o = L.lossk_ce_fwd_bwd(H, W, y, z_weight=1e-3, ws=ws)
    r = L.lossk_ce_fwd_bwd(H, W, y, z_weight=1e-3)
    torch.cuda.synchronize()
    assert torch.equal(o["lse"], r["lse"]) and torch.equal(o["d_weight"], r["d_weight"])
    assert torch.equal(o["d_hidden"], r["d_hidden"]) and torch.equal(o["scalars"], r["scalars"])


def test_all_masked_gives_zeros(L):
    n, d, V = 70, 64, 300
    H = torch.randn(n, d, device="cuda").to(torch.bfloat16)
    W = torch.randn(V, d, device="cuda").to(torch.bfloat16)
    y = torch.randint(0, V, (n,), device="cuda")
    m = torch.zeros(n, dtype=torch.uint8, device="cuda")
    o = L.lossk_ce_fwd_bwd(H, W, y, loss_mask=m, z_weight=0.1)
    torch.cuda.synchronize()
    assert torch.all(o["scalars"] == 0) and torch.all(o["ce"] == 0)
    assert torch.all(o["d_hidden"] == 0) and torch.all(o["d_weight"] == 0)
    assert torch.all(torch.isfinite(o["lse"]))


@pytest.mark.parametrize("dtype", ["bf16", "fp32", "f16"])
def test_vocab_of_one(L, dtype):
    """A single class: CE is zero and its gradient vanishes; only the z term
    (lse^2, gradient 2 w_z lse) remains.  Both the training step and CE from
    given logits, against the oracle."""
    n, d, V = 130, 72, 1
    g = np.random.default_rng(62)
    Hn = li.round_to(g.standard_normal((n, d)).astype(np.float32), dtype)
    Wn = li.round_to((g.standard_normal((V, d)) * 0.3).astype(np.float32), dtype)
    yn = np.zeros(n, np.int64)
    wz, gs = 0.05, 0.75
    out = L.lossk_ce_fwd_bwd(_dev(Hn, dtype), _dev(Wn, dtype), _dev(yn, ""), z_weight=wz, grad_scale=gs)
    torch.cuda.synchronize()
    ref = oracle.ce_fwd(Hn, Wn, yn, z_weight=wz)
    dH, dW = oracle.ce_bwd(Hn, Wn, yn, z_weight=wz, grad_scale=gs)
    lt, gt = _tol(dtype)
    close_loss(_np(out["ce"]), ref["ce"], lt)
    close_loss(_np(out["lse"]), ref["lse"], lt)
    close_loss(_np(out["scalars"]), [ref["total"], ref["ce_mean"], ref["z_mean"]], lt)
    assert rel_l2(_np(out["d_hidden"]), dH) <= gt
    assert rel_l2(_np(out["d_weight"]), dW) <= gt
    X = li.round_to((g.standard_normal((n, V)) * 2).astype(np.float32), dtype)
    o = L.lossk_ce_from_logits(_dev(X, dtype), _dev(yn, ""), z_weight=wz, grad_scale=gs, want_grad=True)
    torch.cuda.synchronize()
    r = oracle.ce_from_logits(X, yn, z_weight=wz, grad_scale=gs, want_grad=True)
    close_loss(_np(o["ce"]), r["ce"], lt)
    close_loss(_np(o["scalars"]), [r["total"], r["ce_mean"], r["z_mean"]], lt)
    assert rel_l2(_np(o["grad_logits"]), _grad_ref(r["grad"], dtype)) <= gt


@pytest.mark.parametrize("dtype", ["bf16", "fp32", "f16"])
@pytest.mark.parametrize("V", [1000, 1003])
def test_distill_from_logits_masked_vocabulary(L, dtype, V):
    """The same vocabulary entries masked out (-inf) in student and teacher rows:
    probability 0 on both sides, so the losses are finite and the gradient is 0
    there; against the oracle, in all three directions, through whole 16-byte
    vectors of -inf (V 1000) and the element-wise path (V 1003)."""
    n = 37
    g = np.random.default_rng(V + 5)
    X = li.round_to((g.standard_normal((n, V)) * 2).astype(np.float32), dtype)
    Tt = li.round_to((g.standard_normal((n, V)) * 3).astype(np.float32), dtype)
    X[:, 0:3] = -np.inf
    X[:, 40:400] = -np.inf
    Tt[:, 0:3] = -np.inf
    Tt[:, 40:400] = -np.inf
    lt, gt = _tol(dtype)
    for direction in ("ce", "fkl", "rkl"):
        o = L.lossk_distill_from_logits(_dev(X, dtype), _dev(Tt, dtype), direction, temperature=1.5,
                                        z_weight=1e-3, want_grad=True)
        torch.cuda.synchronize()
        r = oracle.distill_from_logits(X, Tt, direction, temperature=1.5, z_weight=1e-3)
        assert np.isfinite(_np(o["per_token"])).all() and np.isfinite(_np(o["grad_logits"])).all()
        close_loss(_np(o["per_token"]), r["per_token"], lt)
        close_loss(_np(o["lse"]), r["lse"], lt)
        assert rel_l2(_np(o["grad_logits"]), _grad_ref(r["grad"], dtype)) <= gt
        assert np.all(_np(o["grad_logits"])[:, 40:400] == 0)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("V", [1000, 1003])
@pytest.mark.parametrize("side", ["teacher", "student"])
def test_distill_from_logits_one_sided_mask(L, dtype, V, side):
    """Entries masked out (-inf) on one side only, against the oracle in all three
    directions.  Where only the masked side's probability weights the term
    (teacher zeros in CE and forward KL, student zeros in reverse KL) the loss
    and the gradient are finite and match; where the other side keeps mass on a
    masked entry the loss is +inf in both.  The whole-vector path recomputes
    these rows element-wise (V 1000); V 1003 takes the element-wise path."""
    n = 29
    g = np.random.default_rng(V + 17)
    X = li.round_to((g.standard_normal((n, V)) * 2).astype(np.float32), dtype)
    Tt = li.round_to((g.standard_normal((n, V)) * 3).astype(np.float32), dtype)
    tgt = Tt if side == "teacher" else X
    tgt[:, 5:9] = -np.inf
    tgt[:, 300:360] = -np.inf
    tgt[3, 100] = -np.inf                                   # one more entry in one row
    lt, gt = _tol(dtype)
    for direction in ("ce", "fkl", "rkl"):
        o = L.lossk_distill_from_logits(_dev(X, dtype), _dev(Tt, dtype), direction, temperature=1.5,
                                        z_weight=1e-3, want_grad=True)
        torch.cuda.synchronize()
        r = oracle.distill_from_logits(X, Tt, direction, temperature=1.5, z_weight=1e-3)
        got = _np(o["per_token"])
        if (side == "student") == (direction != "rkl"):
            assert np.all(np.isposinf(r["per_token"])) and np.all(np.isposinf(got))
            continue
        assert np.isfinite(got).all() and np.isfinite(_np(o["grad_logits"])).all()
        close_loss(got, r["per_token"], lt)
        close_loss(_np(o["lse"]), r["lse"], lt)
        assert rel_l2(_np(o["grad_logits"]), _grad_ref(r["grad"], dtype)) <= gt
        if side == "student":
            assert np.all(_np(o["grad_logits"])[:, 300:360] == 0)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("direction", ["ce", "fkl"])
def test_distill_step_teacher_zeros(L, direction, dtype):
    """The distillation training step with teacher logits of -inf on some vocabulary
    entries (probability 0 for the teacher, the student's stays positive): CE and
    forward KL stay finite (0 log 0 = 0 in the teacher's statistics), against the
    oracle, on the tensor-core (bf16) and FFMA (fp32) paths, whose teacher
    statistics recompute such rows with the -inf test.  Reverse KL is +inf there
    by definition."""
    n, d, V = 200, 136, 1032
    x = _inputs("distill_z_4096x2048", seed=13, n_tok=n, d_model=d, vocab=V)
    Tt = x["teacher"].copy()
    Tt[:, 100:300] = -np.inf
    Tt[7, :] = -np.inf
    Tt[7, 5] = 2.0                               # a one-hot teacher row
    H, W = _dev(x["hidden"], dtype), _dev(x["weight"], dtype)
    out = L.lossk_distill_fwd_bwd(H, W, _dev(Tt, dtype), direction, temperature=2.0, z_weight=1e-3)
    torch.cuda.synchronize()
    r = oracle.distill(x["hidden"], x["weight"], Tt, direction, temperature=2.0, z_weight=1e-3)
    lt, gt = _tol(dtype)
    assert np.isfinite(_np(out["per_token"])).all()
    close_loss(_np(out["per_token"]), r["per_token"], lt)
    close_loss(_np(out["scalars"]), [r["total"], r["distill_mean"], r["z_mean"]], lt)
    assert rel_l2(_np(out["d_hidden"]), r["dH"]) <= gt
    assert rel_l2(_np(out["d_weight"]), r["dW"]) <= gt


@pytest.mark.parametrize("dtype", ["bf16", "fp32", "f16"])
@pytest.mark.parametrize("V", [1003, 3000, 70000])
def test_distill_identical_teacher(L, dtype, V):
    """Teacher logits equal to the student's: forward and reverse KL are zero
    per token and their gradients are the z term's alone, against the oracle."""
    n = 40
    X = li.round_to((np.random.default_rng(V).standard_normal((n, V)) * 2).astype(np.float32), dtype)
    lt, gt = _tol(dtype)
    for direction in ("fkl", "rkl"):
        o = L.lossk_distill_from_logits(_dev(X, dtype), _dev(X, dtype), direction, temperature=1.7,
                                        z_weight=0.2, want_grad=True)
        torch.cuda.synchronize()
        r = oracle.distill_from_logits(X, X, direction, temperature=1.7, z_weight=0.2)
        assert np.abs(_np(o["per_token"])).max() <= lt
        close_loss(_np(o["lse"]), r["lse"], lt)
        assert rel_l2(_np(o["grad_logits"]), _grad_ref(r["grad"], dtype)) <= gt


def test_device_status_clean_after_calls(L):
    n, d, V = 64, 64, 256
    ws = L.workspace(L.lossk.KIND_CE_FWD_BWD, n, d, V, 1)
    H = torch.randn(n, d, device="cuda").to(torch.bfloat16)
    W = torch.randn(V, d, device="cuda").to(torch.bfloat16)
    y = torch.randint(0, V, (n,), device="cuda")
    L.lossk_ce_fwd_bwd(H, W, y, ws=ws)
    assert L.lossk_device_status(ws) == 580


# ---------------------------------------------------------------------------
# Gradient accumulation, sum reduction, the chunk self-check, distillation from
# given logits.

@pytest.mark.parametrize("dtype,shape", [("bf16", (300, 256, 2000)), ("bf16", (257, 520, 3000)),
                                         ("fp32", (130, 72, 300)), ("f16", (257, 520, 3000))])
def test_ce_accumulate_and_sum_flags(L, dtype, shape):
    n, d, V = shape
    x = _redraw(_inputs("ce_512x1024x32000", seed=50, n_tok=n, d_model=d, vocab=V), dtype, 1, n, d, V)
    mask = li.mask(3, n, 0.2)
    nv = int(mask.sum())
    wz, gs = 1e-3, 0.75
    H, W, y, m = _dev(x["hidden"], dtype), _dev(x["weight"], dtype), _dev(x["targets"], ""), _dev(mask, "")
    ref = oracle.ce_fwd(x["hidden"], x["weight"], x["targets"], mask=mask, z_weight=wz)
    dH, dW = oracle.ce_bwd(x["hidden"], x["weight"], x["targets"], mask=mask, z_weight=wz, grad_scale=gs)
    lt, gt = _tol(dtype)
    g = torch.Generator(device="cuda").manual_seed(3)
    # starting gradients of the same order as the ones added, so that fp32 keeps the sum exact enough
    h0 = torch.randn(n, d, device="cuda", generator=g) * 1e-4
    w0 = torch.randn(V, d, device="cuda", generator=g) * 1e-3
    for flags in (L.lossk.ACCUMULATE_GRADS, L.lossk.REDUCE_SUM, L.lossk.ACCUMULATE_GRADS | L.lossk.REDUCE_SUM):
        acc, sm = bool(flags & L.lossk.ACCUMULATE_GRADS), bool(flags & L.lossk.REDUCE_SUM)
        dh, dw = h0.clone(), w0.clone()
        o = L.lossk_ce_fwd_bwd_ex(H, W, y, loss_mask=m, chunk=64, z_weight=wz, grad_scale=gs,
                                  flags=flags, d_hidden=dh, d_weight=dw)
        torch.cuda.synchronize()
        k = nv if sm else 1
        close_loss(_np(o["scalars"]), [ref["total"] * k, ref["ce_mean"] * k, ref["z_mean"] * k], lt)
        close_loss(_np(o["lse"]), ref["lse"], lt)
        base_h = _np(h0) if acc else 0.0
        base_w = _np(w0) if acc else 0.0
        assert rel_l2(_np(dh) - base_h, dH * k) <= gt, flags
        assert rel_l2(_np(dw) - base_w, dW * k) <= gt, flags


def test_ce_accumulate_through_the_recompute_fallback(L):
    """A 160-nat row sends the training step to the separate passes; with
    accumulation the caller's gradients must still receive the sum once."""
    n, d, V = 130, 64, 1000
    x = _inputs("ce_512x1024x32000", seed=9, n_tok=n, d_model=d, vocab=V)
    Hn, Wn, yn = x["hidden"].copy(), x["weight"].copy(), x["targets"].copy()
    Hn[7, :] = 1.0
    Wn[3, :] = 2.5
    Wn[5, :] = 0.0
    yn[7] = 5
    Hn, Wn = li.to_bf16_values(Hn), li.to_bf16_values(Wn)
    H, W, y = _dev(Hn, "bf16"), _dev(Wn, "bf16"), _dev(yn, "")
    h0 = torch.full((n, d), 0.25, device="cuda")
    w0 = torch.full((V, d), -0.5, device="cuda")
    dh, dw = h0.clone(), w0.clone()
    L.lossk_ce_fwd_bwd_ex(H, W, y, z_weight=1e-4, flags=L.lossk.ACCUMULATE_GRADS, d_hidden=dh, d_weight=dw)
    torch.cuda.synchronize()
    dH, dW = oracle.ce_bwd(Hn, Wn, yn, z_weight=1e-4)
    assert rel_l2(_np(dh) - 0.25, dH) <= BF16_GRAD
    assert rel_l2(_np(dw) + 0.5, dW) <= BF16_GRAD


@pytest.mark.parametrize("direction", ["ce", "rkl"])
def test_distill_accumulate_and_sum_flags(L, direction):
    n, d, V = 200, 256, 1024
    x = _inputs("distill_z_4096x2048", seed=51, n_tok=n, d_model=d, vocab=V)
    mask = li.mask(6, n, 0.1)
    nv = int(mask.sum())
    r = oracle.distill(x["hidden"], x["weight"], x["teacher"], direction, temperature=2.0, mask=mask,
                       z_weight=1e-3)
    h0 = torch.ones(n, d, device="cuda") * 0.1
    w0 = torch.ones(V, d, device="cuda") * -0.2
    flags = L.lossk.ACCUMULATE_GRADS | L.lossk.REDUCE_SUM
    dh, dw = h0.clone(), w0.clone()
    o = L.lossk_distill_fwd_bwd_ex(_dev(x["hidden"], "bf16"), _dev(x["weight"], "bf16"),
                                   _dev(x["teacher"], "bf16"), direction, temperature=2.0,
                                   loss_mask=_dev(mask, ""), z_weight=1e-3, flags=flags,
                                   d_hidden=dh, d_weight=dw)
    torch.cuda.synchronize()
    close_loss(_np(o["scalars"]), [r["total"] * nv, r["distill_mean"] * nv, r["z_mean"] * nv], BF16_LOSS)
    assert rel_l2(_np(dh) - 0.1, r["dH"] * nv) <= BF16_GRAD
    assert rel_l2(_np(dw) + 0.2, r["dW"] * nv) <= BF16_GRAD


def test_unknown_flag_bits_are_refused(L):
    n, d, V = 64, 64, 512
    H = torch.randn(n, d, device="cuda").to(torch.bfloat16)
    W = torch.randn(V, d, device="cuda").to(torch.bfloat16)
    y = torch.randint(0, V, (n,), device="cuda")
    dh = torch.full((n, d), 3.0, device="cuda")
    with pytest.raises(L.LosskError) as e:
        L.lossk_ce_fwd_bwd_ex(H, W, y, flags=4, d_hidden=dh)
    assert e.value.status == 592
    assert torch.all(dh == 3.0)


@pytest.mark.parametrize("dtype,shape", [("bf16", (300, 256, 2000)), ("fp32", (64, 64, 1000)),
                                         ("bf16", (2048, 1024, 151936)), ("f16", (300, 256, 2000))])
def test_chunk_invariance_self_check(L, dtype, shape):
    n, d, V = shape
    x = _redraw(_inputs("ce_512x1024x32000", seed=52, n_tok=n, d_model=d, vocab=V), dtype, 1, n, d, V)
    delta = L.lossk_ce_chunk_invariance(_dev(x["hidden"], dtype), _dev(x["weight"], dtype),
                                        _dev(x["targets"], ""), loss_mask=_dev(li.mask(2, n, 0.1), ""),
                                        z_weight=1e-3)
    assert delta == 0.0


# V 1003: rows that are not 16-byte multiples (the element-wise loops); 3000:
# fewer 16-byte vectors than threads; 70000: several rounds, the last ragged
@pytest.mark.parametrize("dtype", ["bf16", "fp32", "f16"])
@pytest.mark.parametrize("direction", ["ce", "fkl", "rkl"])
@pytest.mark.parametrize("V", [3000, 1003, 70000])
def test_distill_from_logits(L, dtype, direction, V):
    n = 67
    g = np.random.default_rng(V + len(direction))
    X = li.round_to((g.standard_normal((n, V)) * 2).astype(np.float32), dtype)
    Tt = li.round_to((g.standard_normal((n, V)) * 3).astype(np.float32), dtype)
    mask = li.mask(7, n, 0.15)
    for sm in (False, True):
        r = oracle.distill_from_logits(X, Tt, direction, temperature=1.5, mask=mask, z_weight=1e-3,
                                       grad_scale=0.9, reduce_sum=sm)
        flags = L.lossk.REDUCE_SUM if sm else 0
        o = L.lossk_distill_from_logits(_dev(X, dtype), _dev(Tt, dtype), direction, temperature=1.5,
                                        loss_mask=_dev(mask, ""), z_weight=1e-3, grad_scale=0.9,
                                        flags=flags)
        torch.cuda.synchronize()
        lt, gt = _tol(dtype)
        close_loss(_np(o["per_token"]), r["per_token"], lt)
        close_loss(_np(o["lse"]), r["lse"], lt)
        close_loss(_np(o["scalars"]), [r["total"], r["distill_mean"], r["z_mean"]], lt)
        assert rel_l2(_np(o["grad_logits"]), _grad_ref(r["grad"], dtype)) <= gt
    # accumulation: two calls into a zeroed gradient give twice the gradient
    gl = torch.zeros(n, V, device="cuda", dtype={"bf16": torch.bfloat16, "f16": torch.float16}.get(dtype, torch.float32))
    for _ in range(2):
        L.lossk_distill_from_logits(_dev(X, dtype), _dev(Tt, dtype), direction, temperature=1.5,
                                    loss_mask=_dev(mask, ""), z_weight=1e-3, grad_scale=0.9,
                                    flags=L.lossk.ACCUMULATE_GRADS, grad_logits=gl)
    torch.cuda.synchronize()
    r = oracle.distill_from_logits(X, Tt, direction, temperature=1.5, mask=mask, z_weight=1e-3, grad_scale=0.9)
    if dtype == "f16":
        # what two exact calls accumulated in fp16 hold: round(round(g) + g)
        ideal = _grad_ref(_grad_ref(r["grad"], dtype) + r["grad"], dtype)
    else:
        ideal = 2 * r["grad"]
    assert rel_l2(_np(gl), ideal) <= _tol(dtype)[1]


# ---------------------------------------------------------------------------
# Vocabulary-parallel cross-entropy.  The shards run one after another on one
# GPU; their partials are stacked in shard order, as the all-gather between
# ranks stacks them, then combined; d_hidden is the sum of the shards' shares
# (what the all-reduce between ranks computes) and d_weight their concatenation.
def _shard_step(L, H, W, y, cuts, mask, wz, gs):
    V = W.shape[0]
    edges = [0] + list(cuts) + [V]
    parts, shards = [], []
    for v0, v1 in zip(edges[:-1], edges[1:]):
        Ws = W[v0:v1].contiguous()
        parts.append(L.lossk_ce_shard_fwd(H, Ws, y, v0, V))
        shards.append((v0, Ws))
    pa = torch.stack(parts)
    c = L.lossk_ce_shard_combine(pa, loss_mask=mask, z_weight=wz)
    dh, dws = None, []
    for v0, Ws in shards:
        g = L.lossk_ce_shard_bwd(H, Ws, y, v0, V, c["lse"], loss_mask=mask, z_weight=wz, grad_scale=gs)
        dh = g["d_hidden"] if dh is None else dh + g["d_hidden"]
        dws.append(g["d_weight"])
    torch.cuda.synchronize()
    return pa, c, dh, torch.cat(dws)


@pytest.mark.parametrize("dtype", ["bf16", "fp32", "f16"])
@pytest.mark.parametrize("shape,cuts", [((300, 200, 1000), (8, 504)),       # a one-tile shard
                                        ((130, 1024, 5000), (2500,)),      # two halves
                                        ((257, 520, 2000), (1000, 1001, 1999))])   # one-row shards
def test_vocab_shards_small(L, dtype, shape, cuts):
    n, d, V = shape
    x = _redraw(_inputs("ce_512x1024x32000", seed=41, n_tok=n, d_model=d, vocab=V), dtype, 4, n, d, V)
    yn = x["targets"].copy()
    yn[:3] = [0, V - 1, cuts[0]]                # the vocabulary's ends and a shard's first row
    mask = li.mask(8, n, 0.1)
    wz, gs = 1e-3, 1.5
    H, W, y, m = _dev(x["hidden"], dtype), _dev(x["weight"], dtype), _dev(yn, ""), _dev(mask, "")
    pa, c, dh, dw = _shard_step(L, H, W, y, cuts, m, wz, gs)
    lt, gt = _tol(dtype)
    # each shard's partials against the oracle's
    edges = [0] + list(cuts) + [V]
    for p, (v0, v1) in enumerate(zip(edges[:-1], edges[1:])):
        r = oracle.ce_shard_fwd(x["hidden"], x["weight"][v0:v1], yn, v0, V)
        close_loss(_np(pa[p, 0]), r[0], lt)
        close_loss(_np(pa[p, 1]), r[1], lt)
        assert np.array_equal(_np(pa[p, 2]), r[2])
    ref = oracle.ce_fwd(x["hidden"], x["weight"], yn, mask=mask, z_weight=wz)
    dH, dW = oracle.ce_bwd(x["hidden"], x["weight"], yn, mask=mask, z_weight=wz, grad_scale=gs)
    close_loss(_np(c["lse"]), ref["lse"], lt)
    close_loss(_np(c["ce"]), ref["ce"], lt)
    close_loss(_np(c["scalars"]), [ref["total"], ref["ce_mean"], ref["z_mean"]], lt)
    assert rel_l2(_np(dh), dH) <= gt
    assert rel_l2(_np(dw), dW) <= gt


def test_vocab_shards_qwen3_head_split_in_two(L):
    """The Qwen3 head shape (n 2048, d 1024, V 151936, bf16) split into two
    shards of 75968 rows: every token's lse and the scalars against the
    oracle's full forward, sampled tokens' loss and d_hidden rows, and
    sampled d_weight rows from both shards."""
    w = li.WORKLOADS["qwen3_0p6b_head"]
    x = _inputs(w)
    H, W, y = _dev(x["hidden"], "bf16"), _dev(x["weight"], "bf16"), _dev(x["targets"], "")
    half = w.vocab // 2
    pa, c, dh, dw = _shard_step(L, H, W, y, (half,), None, 0.0, 1.0)
    assert np.array_equal(_np(pa[:, 2]).sum(0), np.ones(w.n_tok))
    full = _qwen3_oracle(x, w)
    close_loss(_np(c["lse"]), full["lse"], BF16_LOSS)
    close_loss(_np(c["ce"]), full["ce"], BF16_LOSS)
    close_loss(_np(c["scalars"]), [full["total"], full["ce_mean"], full["z_mean"]], BF16_LOSS)
    rows = np.sort(np.random.default_rng(17).choice(w.n_tok, 24, replace=False))
    s = oracle.ce_token_rows(x["hidden"], x["weight"], x["targets"], rows)
    assert rel_l2(_np(dh)[rows], s["dH"]) <= BF16_GRAD
    vrows = np.concatenate([np.unique(x["targets"])[:12], [half - 1, half],
                            np.random.default_rng(18).choice(w.vocab, 12, replace=False)])
    dwr = oracle.ce_dweight_rows(x["hidden"], x["weight"], x["targets"], full["lse"], vrows)
    assert rel_l2(_np(dw)[vrows], dwr) <= BF16_GRAD


def test_vocab_shard_combine_refuses_shards_that_do_not_tile(L):
    """A target held by no shard (a shard left out) or by two (a shard given
    twice): 586, and no output written."""
    n, d, V = 64, 64, 512
    x = _inputs("ce_512x1024x32000", seed=43, n_tok=n, d_model=d, vocab=V)
    H, W, y = _dev(x["hidden"], "bf16"), _dev(x["weight"], "bf16"), _dev(x["targets"], "")
    y[0], y[1] = 0, V - 1
    p0 = L.lossk_ce_shard_fwd(H, W[:256].contiguous(), y, 0, V)
    p1 = L.lossk_ce_shard_fwd(H, W[256:].contiguous(), y, 256, V)
    lse = torch.full((n,), -7.0, device="cuda")
    for bad in (torch.stack([p0]), torch.stack([p0, p1, p1])):
        with pytest.raises(L.LosskError) as e:
            L.lossk_ce_shard_combine(bad, lse_out=lse)
        assert e.value.status == 586
    assert bool((lse == -7.0).all())
    c = L.lossk_ce_shard_combine(torch.stack([p0, p1]), lse_out=lse)
    torch.cuda.synchronize()
    close_loss(_np(c["lse"]), oracle.ce_fwd(x["hidden"], x["weight"], _np(y).astype(np.int64))["lse"], BF16_LOSS)
    # a shard outside the vocabulary, and a target outside it
    with pytest.raises(L.LosskError) as e:
        L.lossk_ce_shard_fwd(H, W[:256].contiguous(), y, 300, V)
    assert e.value.status == 582
    y[5] = V
    with pytest.raises(L.LosskError) as e:
        L.lossk_ce_shard_fwd(H, W[:256].contiguous(), y, 0, V)
    assert e.value.status == 586
