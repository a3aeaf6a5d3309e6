"""fp64 CPU oracle for the fused LM-head loss -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never loads it and
shares no code with it: the arithmetic lives in ``lossk_oracle.c`` (plain C,
double precision, ``-ffp-contract=off``), which this module compiles with gcc
on first use and calls through ctypes.  ``brute.py`` restates the same
definitions as pure-Python loops for tiny inputs.

Every function cites the passage it follows in the C source.  Inputs are
numpy arrays holding the exact values the GPU receives (bf16 or fp32 values
widened to float32); outputs are float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lossk_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liblossk_oracle.so")
_lock = threading.Lock()
_lib = None

DIRECTIONS = {"ce": 0, "fkl": 1, "rkl": 2}


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liblossk_oracle.so``."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, dbl, vp, i32 = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
            lib.oracle_status_name.restype = ctypes.c_char_p
            lib.oracle_status_name.argtypes = [i32]
            lib.oracle_work_fits.argtypes = [i64, i64, i64, i64]
            lib.oracle_dims_check.argtypes = [i64, i64, i64]
            lib.oracle_chunk_check.argtypes = [i64, i64]
            lib.oracle_logit_cells.restype = dbl
            lib.oracle_logit_cells.argtypes = [i64, i64]
            lib.oracle_targets_in_range.argtypes = [vp, i64, i64]
            lib.oracle_peak_logit_cells.argtypes = [i64, i64, i64, vp, vp]
            lib.oracle_ce_from_logits.argtypes = [vp, vp, vp, i64, i64, dbl, dbl, vp, vp, vp, vp]
            lib.oracle_ce_fwd.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, dbl, vp, vp, vp]
            lib.oracle_ce_bwd.argtypes = [vp, vp, vp, vp, i64, i64, i64, dbl, dbl, vp, vp]
            lib.oracle_ce_token_rows.argtypes = [vp, vp, vp, vp, i64, i64, i64, dbl, dbl,
                                                 vp, i64, vp, vp, vp]
            lib.oracle_ce_dweight_rows.argtypes = [vp, vp, vp, vp, i64, i64, i64, dbl, dbl,
                                                   vp, vp, i64, vp]
            lib.oracle_distill.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i32, dbl, dbl,
                                           dbl, vp, vp, vp, vp, vp]
            lib.oracle_distill_from_logits.argtypes = [vp, vp, vp, i64, i64, i32, dbl, dbl, dbl, i32,
                                                        vp, vp, vp, vp]
            lib.oracle_distill_token_rows.argtypes = [vp, vp, vp, vp, i64, i64, i64, i32, dbl,
                                                      dbl, dbl, vp, i64, vp, vp, vp]
            lib.oracle_ce_shard_fwd.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, vp]
            lib.oracle_ce_shard_combine.argtypes = [vp, i64, i64, vp, dbl, vp, vp, vp]
            lib.oracle_ce_shard_bwd.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, dbl, dbl,
                                                vp, vp, vp]
            lib.oracle_reduce_tokens.argtypes = [vp, vp, vp, i64, dbl, vp]
            lib.oracle_distill_dweight_rows.argtypes = [vp, vp, vp, vp, i64, i64, i64, i32, dbl,
                                                        dbl, dbl, vp, vp, vp, i64, vp]
            _lib = lib
    return _lib


class OracleError(RuntimeError):
    def __init__(self, status: int):
        super().__init__(f"oracle refused: {status} ({status_name(status)})")
        self.status = status


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _i64(a):
    return np.ascontiguousarray(a, dtype=np.int64)


def _mask(m):
    return None if m is None else np.ascontiguousarray(m, dtype=np.uint8)


def _p(a):
    return None if a is None else a.ctypes.data


# ---- contract (integer / host arithmetic) -----------------------------------

def status_name(code: int) -> str:
    return _load().oracle_status_name(int(code)).decode()


def work_fits(n, d, V, ceiling) -> bool:
    return bool(_load().oracle_work_fits(n, d, V, ceiling))


def dims_check(n, d, V) -> int:
    return _load().oracle_dims_check(n, d, V)


def chunk_check(chunk, V) -> int:
    return _load().oracle_chunk_check(chunk, V)


def logit_cells(chunk, V) -> float:
    return _load().oracle_logit_cells(chunk, V)


def targets_in_range(y, n, V) -> bool:
    y = _i64(y)
    return bool(_load().oracle_targets_in_range(_p(y), n, V))


def peak_logit_cells(n, V, chunk) -> dict:
    out = np.zeros(3, np.float64)
    nch = np.zeros(1, np.int64)
    st = _load().oracle_peak_logit_cells(n, V, chunk, _p(out), _p(nch))
    return {"chunked_cells": float(out[0]), "materialized_cells": float(out[1]),
            "ratio": float(out[2]), "n_chunks": int(nch[0]), "status": int(st)}


# ---- losses ------------------------------------------------------------------

def ce_from_logits(logits, targets, mask=None, z_weight=0.0, grad_scale=1.0, want_grad=False):
    """Cross-entropy from materialised logits [n][V] (see oracle_ce_from_logits)."""
    x = _f32(logits)
    n, V = x.shape
    y, m = _i64(targets), _mask(mask)
    lse, ce = np.zeros(n), np.zeros(n)
    scal = np.zeros(3)
    grad = np.zeros((n, V)) if want_grad else None
    st = _load().oracle_ce_from_logits(_p(x), _p(y), _p(m), n, V, z_weight, grad_scale,
                                       _p(lse), _p(ce), _p(scal), _p(grad))
    if st != 580:
        raise OracleError(st)
    return {"lse": lse, "ce": ce, "total": scal[0], "ce_mean": scal[1], "z_mean": scal[2],
            "grad": grad}


def ce_fwd(H, W, targets, mask=None, chunk=None, z_weight=0.0):
    """Fused projection + chunked cross-entropy (see oracle_ce_fwd)."""
    H, W = _f32(H), _f32(W)
    n, d = H.shape
    V = W.shape[0]
    y, m = _i64(targets), _mask(mask)
    chunk = n if chunk is None else chunk
    lse, ce, scal = np.zeros(n), np.zeros(n), np.zeros(3)
    st = _load().oracle_ce_fwd(_p(H), _p(W), _p(y), _p(m), n, d, V, chunk, z_weight,
                               _p(lse), _p(ce), _p(scal))
    if st != 580:
        raise OracleError(st)
    return {"lse": lse, "ce": ce, "total": scal[0], "ce_mean": scal[1], "z_mean": scal[2]}


def ce_bwd(H, W, targets, mask=None, z_weight=0.0, grad_scale=1.0):
    """Analytic backward of the fused loss (see oracle_ce_bwd)."""
    H, W = _f32(H), _f32(W)
    n, d = H.shape
    V = W.shape[0]
    y, m = _i64(targets), _mask(mask)
    dH, dW = np.zeros((n, d)), np.zeros((V, d))
    st = _load().oracle_ce_bwd(_p(H), _p(W), _p(y), _p(m), n, d, V, z_weight, grad_scale,
                               _p(dH), _p(dW))
    if st != 580:
        raise OracleError(st)
    return dH, dW


def ce_token_rows(H, W, targets, rows, mask=None, z_weight=0.0, grad_scale=1.0, want_dh=True):
    """lse, target logit and dH for the listed tokens only."""
    H, W = _f32(H), _f32(W)
    n, d = H.shape
    V = W.shape[0]
    y, m, r = _i64(targets), _mask(mask), _i64(rows)
    k = r.shape[0]
    lse, tgt = np.zeros(k), np.zeros(k)
    dh = np.zeros((k, d)) if want_dh else None
    st = _load().oracle_ce_token_rows(_p(H), _p(W), _p(y), _p(m), n, d, V, z_weight,
                                      grad_scale, _p(r), k, _p(lse), _p(tgt), _p(dh))
    if st != 580:
        raise OracleError(st)
    return {"lse": lse, "tgt": tgt, "dH": dh}


def ce_dweight_rows(H, W, targets, lse_all, vrows, mask=None, z_weight=0.0, grad_scale=1.0):
    """dW for the listed vocabulary rows, given every token's oracle lse."""
    H, W = _f32(H), _f32(W)
    n, d = H.shape
    V = W.shape[0]
    y, m, r = _i64(targets), _mask(mask), _i64(vrows)
    lse_all = np.ascontiguousarray(lse_all, dtype=np.float64)
    out = np.zeros((r.shape[0], d))
    st = _load().oracle_ce_dweight_rows(_p(H), _p(W), _p(y), _p(m), n, d, V, z_weight,
                                        grad_scale, _p(lse_all), _p(r), r.shape[0], _p(out))
    if st != 580:
        raise OracleError(st)
    return out


def distill(H, W, teacher, direction, temperature=1.0, mask=None, chunk=None, z_weight=0.0,
            grad_scale=1.0, want_grad=True):
    """Distillation loss and gradients (see oracle_distill)."""
    H, W, Tt = _f32(H), _f32(W), _f32(teacher)
    n, d = H.shape
    V = W.shape[0]
    m = _mask(mask)
    chunk = n if chunk is None else chunk
    dirn = DIRECTIONS[direction] if isinstance(direction, str) else int(direction)
    per, lse, scal = np.zeros(n), np.zeros(n), np.zeros(3)
    dH = np.zeros((n, d)) if want_grad else None
    dW = np.zeros((V, d)) if want_grad else None
    st = _load().oracle_distill(_p(H), _p(W), _p(Tt), _p(m), n, d, V, chunk, dirn,
                                temperature, z_weight, grad_scale, _p(per), _p(lse), _p(scal),
                                _p(dH), _p(dW))
    if st != 580:
        raise OracleError(st)
    return {"per_token": per, "lse": lse, "total": scal[0], "distill_mean": scal[1],
            "z_mean": scal[2], "dH": dH, "dW": dW}


def distill_from_logits(logits, teacher, direction, temperature=1.0, mask=None, z_weight=0.0,
                        grad_scale=1.0, reduce_sum=False, want_grad=True):
    """Distillation from given student logits [n][V] (see oracle_distill_from_logits)."""
    X, Tt = _f32(logits), _f32(teacher)
    n, V = X.shape
    m = _mask(mask)
    dirn = DIRECTIONS[direction] if isinstance(direction, str) else int(direction)
    per, lse, scal = np.zeros(n), np.zeros(n), np.zeros(3)
    grad = np.zeros((n, V)) if want_grad else None
    st = _load().oracle_distill_from_logits(_p(X), _p(Tt), _p(m), n, V, dirn, temperature, z_weight,
                                            grad_scale, 1 if reduce_sum else 0, _p(per), _p(lse),
                                            _p(scal), _p(grad))
    if st != 580:
        raise OracleError(st)
    return {"per_token": per, "lse": lse, "total": scal[0], "distill_mean": scal[1],
            "z_mean": scal[2], "grad": grad}


def distill_token_rows(H, W, teacher, direction, rows, temperature=1.0, mask=None,
                       z_weight=0.0, grad_scale=1.0, want_dh=True):
    """Per listed token: distillation loss, student lse(s/T) and dH row."""
    H, W, Tt = _f32(H), _f32(W), _f32(teacher)
    n, d = H.shape
    V = W.shape[0]
    m, r = _mask(mask), _i64(rows)
    dirn = DIRECTIONS[direction] if isinstance(direction, str) else int(direction)
    k = r.shape[0]
    loss, lse = np.zeros(k), np.zeros(k)
    dh = np.zeros((k, d)) if want_dh else None
    st = _load().oracle_distill_token_rows(_p(H), _p(W), _p(Tt), _p(m), n, d, V, dirn,
                                           temperature, z_weight, grad_scale, _p(r), k,
                                           _p(loss), _p(lse), _p(dh))
    if st != 580:
        raise OracleError(st)
    return {"loss": loss, "lse": lse, "dH": dh}


def distill_dweight_rows(H, W, teacher, direction, lse_all, loss_all, vrows, temperature=1.0,
                         mask=None, z_weight=0.0, grad_scale=1.0):
    """dW for the listed vocabulary rows, given every token's oracle lse(s/T)
    and distillation loss (see oracle_distill_dweight_rows)."""
    H, W, Tt = _f32(H), _f32(W), _f32(teacher)
    n, d = H.shape
    V = W.shape[0]
    m, r = _mask(mask), _i64(vrows)
    dirn = DIRECTIONS[direction] if isinstance(direction, str) else int(direction)
    lse_all = np.ascontiguousarray(lse_all, dtype=np.float64)
    loss_all = np.ascontiguousarray(loss_all, dtype=np.float64)
    out = np.zeros((r.shape[0], d))
    st = _load().oracle_distill_dweight_rows(_p(H), _p(W), _p(Tt), _p(m), n, d, V, dirn,
                                             temperature, z_weight, grad_scale, _p(lse_all),
                                             _p(loss_all), _p(r), r.shape[0], _p(out))
    if st != 580:
        raise OracleError(st)
    return out


def reduce_tokens(loss, lse, mask=None, z_weight=0.0):
    """{total, loss mean, z mean} of per-token values (see oracle_reduce_tokens)."""
    loss = np.ascontiguousarray(loss, dtype=np.float64)
    lse = np.ascontiguousarray(lse, dtype=np.float64)
    m = _mask(mask)
    scal = np.zeros(3)
    st = _load().oracle_reduce_tokens(_p(loss), _p(lse), _p(m), loss.shape[0], z_weight, _p(scal))
    if st != 580:
        raise OracleError(st)
    return {"total": scal[0], "loss_mean": scal[1], "z_mean": scal[2]}


# ---- vocabulary-parallel cross-entropy (see oracle_ce_shard_fwd) ---------------

def ce_shard_fwd(H, W_shard, targets, v0, vocab_total):
    """Partials [3][n] of one vocabulary shard: lse over the shard, the target
    logit if the shard holds the target (else 0), and that 1/0 flag."""
    H, Ws = _f32(H), _f32(W_shard)
    n, d = H.shape
    Vs = Ws.shape[0]
    y = _i64(targets)
    out = np.zeros((3, n))
    st = _load().oracle_ce_shard_fwd(_p(H), _p(Ws), _p(y), n, d, Vs, v0, vocab_total, _p(out))
    if st != 580:
        raise OracleError(st)
    return out


def ce_shard_combine(partials_all, mask=None, z_weight=0.0):
    """lse, ce and the three scalars from the shards' partials [P][3][n]."""
    pa = np.ascontiguousarray(partials_all, dtype=np.float64)
    P, _, n = pa.shape
    m = _mask(mask)
    lse, ce, scal = np.zeros(n), np.zeros(n), np.zeros(3)
    st = _load().oracle_ce_shard_combine(_p(pa), P, n, _p(m), z_weight, _p(lse), _p(ce), _p(scal))
    if st != 580:
        raise OracleError(st)
    return {"lse": lse, "ce": ce, "total": scal[0], "ce_mean": scal[1], "z_mean": scal[2]}


def ce_shard_bwd(H, W_shard, targets, v0, vocab_total, lse_all, mask=None, z_weight=0.0,
                 grad_scale=1.0):
    """The shard's share of d_hidden [n][d] and its d_weight rows [Vs][d]."""
    H, Ws = _f32(H), _f32(W_shard)
    n, d = H.shape
    Vs = Ws.shape[0]
    y, m = _i64(targets), _mask(mask)
    lse_all = np.ascontiguousarray(lse_all, dtype=np.float64)
    dh, dw = np.zeros((n, d)), np.zeros((Vs, d))
    st = _load().oracle_ce_shard_bwd(_p(H), _p(Ws), _p(y), _p(m), n, d, Vs, v0, vocab_total,
                                     z_weight, grad_scale, _p(lse_all), _p(dh), _p(dw))
    if st != 580:
        raise OracleError(st)
    return dh, dw
