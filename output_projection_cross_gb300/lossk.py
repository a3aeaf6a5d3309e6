"""Python binding of liblossk.so: same names as the C ABI, argument marshalling only.

Every function takes torch tensors (device memory allocated by the caller or,
for outputs left as ``None``, by this binding through torch), passes their
pointers and element counts to the C entry point on the current CUDA stream,
and raises :class:`LosskError` for any status other than 580.  All arithmetic
runs in the library's CUDA kernels; there is no fallback of any kind, and
importing this module fails if the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

_i64, _i32, _dbl, _vp, _u32 = ctypes.c_int64, ctypes.c_int32, ctypes.c_double, ctypes.c_void_p, ctypes.c_uint32

F32, BF16, F16 = 0, 1, 2
KIND_CE_FWD, KIND_CE_BWD, KIND_CE_FWD_BWD, KIND_FROM_LOGITS, KIND_DISTILL, KIND_CE_CHUNK_CHECK = 0, 1, 2, 3, 4, 5
KIND_SHARD_FWD, KIND_SHARD_BWD, KIND_SHARD_COMBINE = 6, 7, 8
ACCUMULATE_GRADS, REDUCE_SUM = 1, 2
DIRECTIONS = {"ce": 0, "fkl": 1, "rkl": 2}
OK = 580


class lossk_peak_cells(ctypes.Structure):
    _fields_ = [("chunked_cells", _dbl), ("materialized_cells", _dbl), ("ratio", _dbl),
                ("n_chunks", _i64), ("status", _i32)]


def _load():
    path = _build.LIB
    if not os.path.exists(path):
        raise ImportError(
            f"liblossk.so is not built ({path}); run `python -c \"import __graft_entry__ as g; "
            f"g.build()\"` or `python output_projection_cross_gb300/build.py`")
    lib = ctypes.CDLL(path)
    sig = {
        "lossk_status_name": (ctypes.c_char_p, [_i32]),
        "lossk_dims_check": (_i32, [_i64, _i64, _i64]),
        "lossk_chunk_check": (_i32, [_i64, _i64]),
        "lossk_logit_cells": (_dbl, [_i64, _i64]),
        "lossk_work_fits": (_i32, [_i64, _i64, _i64, _i64]),
        "lossk_peak_logit_cells": (_i32, [_i64, _i64, _i64, ctypes.POINTER(lossk_peak_cells)]),
        "lossk_workspace_bytes": (_i64, [_i32, _i64, _i64, _i64, _i32]),
        "lossk_targets_check": (_i32, [_i64, _i64, _vp, _i64, _vp, _i64, _vp]),
        "lossk_ce_fwd": (_i32, [_i64, _i64, _i64, _i64, _i32, _vp, _i64, _vp, _i64, _vp, _i64, _vp,
                                _dbl, _vp, _vp, _vp, _vp, _i64, _vp]),
        "lossk_ce_bwd": (_i32, [_i64, _i64, _i64, _i32, _vp, _i64, _vp, _i64, _vp, _i64, _vp, _dbl,
                                _dbl, _vp, _i64, _vp, _vp, _vp, _i64, _vp]),
        "lossk_ce_fwd_bwd": (_i32, [_i64, _i64, _i64, _i64, _i32, _vp, _i64, _vp, _i64, _vp, _i64,
                                    _vp, _dbl, _dbl, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _vp]),
        "lossk_ce_from_logits": (_i32, [_i64, _i64, _i32, _vp, _i64, _vp, _i64, _vp, _dbl, _dbl,
                                        _vp, _vp, _vp, _vp, _i64, _vp, _i64, _vp]),
        "lossk_distill_fwd_bwd": (_i32, [_i64, _i64, _i64, _i64, _i32, _vp, _i64, _vp, _i64, _vp,
                                         _i64, _vp, _i32, _dbl, _dbl, _dbl, _vp, _vp, _vp, _vp,
                                         _vp, _vp, _i64, _vp]),
        "lossk_ce_fwd_bwd_ex": (_i32, [_i64, _i64, _i64, _i64, _i32, _vp, _i64, _vp, _i64, _vp, _i64,
                                       _vp, _dbl, _dbl, _u32, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _vp]),
        "lossk_distill_fwd_bwd_ex": (_i32, [_i64, _i64, _i64, _i64, _i32, _vp, _i64, _vp, _i64, _vp,
                                            _i64, _vp, _i32, _dbl, _dbl, _dbl, _u32, _vp, _vp, _vp, _vp,
                                            _vp, _vp, _i64, _vp]),
        "lossk_ce_chunk_invariance": (_i32, [_i64, _i64, _i64, _i32, _vp, _i64, _vp, _i64, _vp, _i64,
                                             _vp, _dbl, ctypes.POINTER(_dbl), _vp, _i64, _vp]),
        "lossk_distill_from_logits": (_i32, [_i64, _i64, _i32, _vp, _i64, _vp, _i64, _vp, _i32, _dbl,
                                             _dbl, _dbl, _u32, _vp, _vp, _vp, _vp, _i64, _vp, _i64,
                                             _vp]),
        "lossk_device_status": (_i32, [_vp, _i64, _vp]),
        "lossk_ce_from_logits_static": (_i32, [_i64, _i64, _i32, _vp, _i64, _vp, _i64, _vp, _dbl,
                                               _dbl, _vp, _vp, _vp, _vp, _i64, _vp]),
        "lossk_ce_shard_fwd": (_i32, [_i64, _i64, _i64, _i64, _i64, _i32, _vp, _i64, _vp, _i64, _vp, _i64,
                                      _vp, _i64, _vp, _i64, _vp]),
        "lossk_ce_shard_combine": (_i32, [_i64, _i64, _vp, _i64, _vp, _dbl, _vp, _vp, _vp, _vp, _i64, _vp]),
        "lossk_ce_shard_bwd": (_i32, [_i64, _i64, _i64, _i64, _i64, _i32, _vp, _i64, _vp, _i64, _vp, _i64,
                                      _vp, _dbl, _dbl, _vp, _i64, _vp, _vp, _vp, _i64, _vp]),
        "lossk_selftest_wait": (_i32, [_i32, _i32, _i64, ctypes.POINTER(_i32), _vp, _i64, _vp]),
        "lossk_kernel_name": (ctypes.c_char_p, [_i32]),
        "lossk_launch_count": (_i64, []),
        "lossk_profile_enable": (_i32, [_i32]),
        "lossk_profile_read": (_i32, [ctypes.POINTER(_dbl), ctypes.POINTER(_i64), _i32, _i32]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


lib = _load()
EXPORTED = ("lossk_status_name", "lossk_dims_check", "lossk_chunk_check", "lossk_logit_cells",
            "lossk_work_fits", "lossk_peak_logit_cells", "lossk_workspace_bytes",
            "lossk_targets_check", "lossk_ce_fwd", "lossk_ce_bwd", "lossk_ce_fwd_bwd",
            "lossk_ce_from_logits", "lossk_distill_fwd_bwd", "lossk_device_status",
            "lossk_ce_fwd_bwd_ex", "lossk_distill_fwd_bwd_ex", "lossk_ce_chunk_invariance",
            "lossk_distill_from_logits",
            "lossk_ce_from_logits_static", "lossk_selftest_wait", "lossk_ce_shard_fwd",
            "lossk_ce_shard_combine", "lossk_ce_shard_bwd", "lossk_kernel_name", "lossk_launch_count", "lossk_profile_enable", "lossk_profile_read")
N_KERNELS = 23


class LosskError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: status {status} ({lossk_status_name(status)})")
        self.status = status


def _check(st: int, where: str) -> None:
    if st != OK:
        raise LosskError(st, where)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _len(t):
    return 0 if t is None else t.numel()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float16:
        return F16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype}: bf16, fp16 or fp32")


def _contig(t, name):
    if t is not None and (not t.is_cuda or not t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    return t


# ---- contract -----------------------------------------------------------------

def lossk_status_name(code: int) -> str:
    return lib.lossk_status_name(code).decode()


def lossk_dims_check(n_tok: int, d_model: int, vocab: int) -> int:
    return lib.lossk_dims_check(n_tok, d_model, vocab)


def lossk_chunk_check(chunk: int, vocab: int) -> int:
    return lib.lossk_chunk_check(chunk, vocab)


def lossk_logit_cells(chunk: int, vocab: int) -> float:
    return lib.lossk_logit_cells(chunk, vocab)


def lossk_work_fits(n_tok: int, d_model: int, vocab: int, ceiling: int) -> bool:
    return bool(lib.lossk_work_fits(n_tok, d_model, vocab, ceiling))


def lossk_peak_logit_cells(n_tok: int, vocab: int, chunk: int) -> dict:
    out = lossk_peak_cells()
    lib.lossk_peak_logit_cells(n_tok, vocab, chunk, ctypes.byref(out))
    return {"chunked_cells": out.chunked_cells, "materialized_cells": out.materialized_cells,
            "ratio": out.ratio, "n_chunks": out.n_chunks, "status": out.status}


def lossk_workspace_bytes(kind: int, n_tok: int, d_model: int, vocab: int, dtype: int) -> int:
    return lib.lossk_workspace_bytes(kind, n_tok, d_model, vocab, dtype)


def workspace(kind: int, n_tok: int, d_model: int, vocab: int, dtype: int, device=None):
    nb = lossk_workspace_bytes(kind, n_tok, d_model, vocab, dtype)
    if nb < 0:
        raise LosskError(lossk_dims_check(n_tok, d_model, vocab), "lossk_workspace_bytes")
    return torch.zeros(nb, dtype=torch.uint8, device=device or "cuda")


# ---- device calls -----------------------------------------------------------------

def lossk_targets_check(targets, vocab, ws=None, stream=None) -> int:
    _contig(targets, "targets")
    ws = ws if ws is not None else torch.zeros(256, dtype=torch.uint8, device=targets.device)
    return lib.lossk_targets_check(targets.numel(), vocab, _ptr(targets), targets.numel(),
                                   _ptr(ws), ws.numel(), _stream(stream))


def _ws(ws, kind, n, d, V, dtype, dev):
    return ws if ws is not None else workspace(kind, n, d, V, dtype, dev)


def lossk_ce_fwd(hidden, weight, targets, loss_mask=None, chunk=None, z_weight=0.0, lse_out=None,
                 ce_out=None, scalars_out=None, ws=None, stream=None):
    for t, nm in ((hidden, "hidden"), (weight, "weight"), (targets, "targets"), (loss_mask, "loss_mask")):
        _contig(t, nm)
    n, d = hidden.shape
    V = weight.shape[0]
    dt = _dtype_code(hidden)
    dev = hidden.device
    lse_out = lse_out if lse_out is not None else torch.empty(n, dtype=torch.float32, device=dev)
    ce_out = ce_out if ce_out is not None else torch.empty(n, dtype=torch.float32, device=dev)
    scalars_out = scalars_out if scalars_out is not None else torch.empty(3, dtype=torch.float64, device=dev)
    ws = _ws(ws, KIND_CE_FWD, n, d, V, dt, dev)
    st = lib.lossk_ce_fwd(n, d, V, n if chunk is None else chunk, dt, _ptr(hidden), _len(hidden),
                          _ptr(weight), _len(weight), _ptr(targets), _len(targets), _ptr(loss_mask),
                          z_weight, _ptr(lse_out), _ptr(ce_out), _ptr(scalars_out), _ptr(ws),
                          ws.numel(), _stream(stream))
    _check(st, "lossk_ce_fwd")
    return {"lse": lse_out, "ce": ce_out, "scalars": scalars_out}


def lossk_ce_bwd(hidden, weight, targets, lse, loss_mask=None, z_weight=0.0, grad_scale=1.0,
                 d_hidden=None, d_weight=None, want_d_hidden=True, want_d_weight=True, ws=None,
                 stream=None):
    for t, nm in ((hidden, "hidden"), (weight, "weight"), (targets, "targets"), (lse, "lse"),
                  (loss_mask, "loss_mask")):
        _contig(t, nm)
    n, d = hidden.shape
    V = weight.shape[0]
    dt = _dtype_code(hidden)
    dev = hidden.device
    if want_d_hidden and d_hidden is None:
        d_hidden = torch.empty(n, d, dtype=torch.float32, device=dev)
    if want_d_weight and d_weight is None:
        d_weight = torch.empty(V, d, dtype=torch.float32, device=dev)
    ws = _ws(ws, KIND_CE_BWD, n, d, V, dt, dev)
    st = lib.lossk_ce_bwd(n, d, V, dt, _ptr(hidden), _len(hidden), _ptr(weight), _len(weight),
                          _ptr(targets), _len(targets), _ptr(loss_mask), z_weight, grad_scale,
                          _ptr(lse), _len(lse), _ptr(d_hidden), _ptr(d_weight), _ptr(ws), ws.numel(),
                          _stream(stream))
    _check(st, "lossk_ce_bwd")
    return {"d_hidden": d_hidden, "d_weight": d_weight}


def lossk_ce_fwd_bwd(hidden, weight, targets, loss_mask=None, chunk=None, z_weight=0.0,
                     grad_scale=1.0, lse_out=None, ce_out=None, scalars_out=None, d_hidden=None,
                     d_weight=None, want_d_hidden=True, want_d_weight=True, ws=None, stream=None):
    return lossk_ce_fwd_bwd_ex(hidden, weight, targets, loss_mask, chunk, z_weight, grad_scale, 0,
                               lse_out, ce_out, scalars_out, d_hidden, d_weight, want_d_hidden,
                               want_d_weight, ws, stream)


def lossk_ce_fwd_bwd_ex(hidden, weight, targets, loss_mask=None, chunk=None, z_weight=0.0,
                        grad_scale=1.0, flags=0, lse_out=None, ce_out=None, scalars_out=None,
                        d_hidden=None, d_weight=None, want_d_hidden=True, want_d_weight=True,
                        ws=None, stream=None):
    """flags: ACCUMULATE_GRADS (add into d_hidden / d_weight; outputs created here start at
    zero) and/or REDUCE_SUM.  flags == 0 calls the plain C entry point."""
    for t, nm in ((hidden, "hidden"), (weight, "weight"), (targets, "targets"), (loss_mask, "loss_mask")):
        _contig(t, nm)
    n, d = hidden.shape
    V = weight.shape[0]
    dt = _dtype_code(hidden)
    dev = hidden.device
    lse_out = lse_out if lse_out is not None else torch.empty(n, dtype=torch.float32, device=dev)
    ce_out = ce_out if ce_out is not None else torch.empty(n, dtype=torch.float32, device=dev)
    scalars_out = scalars_out if scalars_out is not None else torch.empty(3, dtype=torch.float64, device=dev)
    alloc = torch.zeros if flags & ACCUMULATE_GRADS else torch.empty
    if want_d_hidden and d_hidden is None:
        d_hidden = alloc(n, d, dtype=torch.float32, device=dev)
    if want_d_weight and d_weight is None:
        d_weight = alloc(V, d, dtype=torch.float32, device=dev)
    ws = _ws(ws, KIND_CE_FWD_BWD, n, d, V, dt, dev)
    args = (_ptr(hidden), _len(hidden), _ptr(weight), _len(weight), _ptr(targets), _len(targets),
            _ptr(loss_mask), z_weight, grad_scale)
    outs = (_ptr(lse_out), _ptr(ce_out), _ptr(scalars_out), _ptr(d_hidden), _ptr(d_weight), _ptr(ws),
            ws.numel(), _stream(stream))
    c = n if chunk is None else chunk
    if flags == 0:
        st = lib.lossk_ce_fwd_bwd(n, d, V, c, dt, *args, *outs)
        _check(st, "lossk_ce_fwd_bwd")
    else:
        st = lib.lossk_ce_fwd_bwd_ex(n, d, V, c, dt, *args, flags, *outs)
        _check(st, "lossk_ce_fwd_bwd_ex")
    return {"lse": lse_out, "ce": ce_out, "scalars": scalars_out, "d_hidden": d_hidden,
            "d_weight": d_weight}


def lossk_ce_from_logits(logits, targets, loss_mask=None, z_weight=0.0, grad_scale=1.0,
                         want_grad=False, lse_out=None, ce_out=None, scalars_out=None,
                         grad_logits=None, ws=None, stream=None):
    for t, nm in ((logits, "logits"), (targets, "targets"), (loss_mask, "loss_mask")):
        _contig(t, nm)
    n, V = logits.shape
    dt = _dtype_code(logits)
    dev = logits.device
    lse_out = lse_out if lse_out is not None else torch.empty(n, dtype=torch.float32, device=dev)
    ce_out = ce_out if ce_out is not None else torch.empty(n, dtype=torch.float32, device=dev)
    scalars_out = scalars_out if scalars_out is not None else torch.empty(3, dtype=torch.float64, device=dev)
    if want_grad and grad_logits is None:
        grad_logits = torch.empty_like(logits)
    ws = _ws(ws, KIND_FROM_LOGITS, n, 1, V, dt, dev)
    st = lib.lossk_ce_from_logits(n, V, dt, _ptr(logits), _len(logits), _ptr(targets),
                                  _len(targets), _ptr(loss_mask), z_weight, grad_scale,
                                  _ptr(lse_out), _ptr(ce_out), _ptr(scalars_out), _ptr(grad_logits),
                                  _len(grad_logits), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "lossk_ce_from_logits")
    return {"lse": lse_out, "ce": ce_out, "scalars": scalars_out, "grad_logits": grad_logits}


def lossk_ce_from_logits_static(logits, targets, loss_mask=None, z_weight=0.0, grad_scale=1.0,
                                want_grad=False, lse_out=None, ce_out=None, scalars_out=None,
                                grad_logits=None, stream=None):
    """lossk_ce_from_logits without a workspace: scratch lives in a device array built
    into the library (n_tok <= 16384).  Outputs left as None are created here with torch;
    a caller that must not allocate passes them all in."""
    for t, nm in ((logits, "logits"), (targets, "targets"), (loss_mask, "loss_mask")):
        _contig(t, nm)
    n, V = logits.shape
    dt = _dtype_code(logits)
    dev = logits.device
    lse_out = lse_out if lse_out is not None else torch.empty(n, dtype=torch.float32, device=dev)
    ce_out = ce_out if ce_out is not None else torch.empty(n, dtype=torch.float32, device=dev)
    scalars_out = scalars_out if scalars_out is not None else torch.empty(3, dtype=torch.float64, device=dev)
    if want_grad and grad_logits is None:
        grad_logits = torch.empty_like(logits)
    st = lib.lossk_ce_from_logits_static(n, V, dt, _ptr(logits), _len(logits), _ptr(targets),
                                         _len(targets), _ptr(loss_mask), z_weight, grad_scale,
                                         _ptr(lse_out), _ptr(ce_out), _ptr(scalars_out),
                                         _ptr(grad_logits), _len(grad_logits), _stream(stream))
    _check(st, "lossk_ce_from_logits_static")
    return {"lse": lse_out, "ce": ce_out, "scalars": scalars_out, "grad_logits": grad_logits}


def lossk_distill_fwd_bwd(hidden, weight, teacher_logits, direction="fkl", temperature=1.0,
                          loss_mask=None, chunk=None, z_weight=0.0, grad_scale=1.0,
                          scalars_out=None, per_token_out=None, lse_out=None, d_hidden=None,
                          d_weight=None, want_d_hidden=True, want_d_weight=True, ws=None,
                          stream=None):
    return lossk_distill_fwd_bwd_ex(hidden, weight, teacher_logits, direction, temperature,
                                    loss_mask, chunk, z_weight, grad_scale, 0, scalars_out,
                                    per_token_out, lse_out, d_hidden, d_weight, want_d_hidden,
                                    want_d_weight, ws, stream)


def lossk_distill_fwd_bwd_ex(hidden, weight, teacher_logits, direction="fkl", temperature=1.0,
                             loss_mask=None, chunk=None, z_weight=0.0, grad_scale=1.0, flags=0,
                             scalars_out=None, per_token_out=None, lse_out=None, d_hidden=None,
                             d_weight=None, want_d_hidden=True, want_d_weight=True, ws=None,
                             stream=None):
    for t, nm in ((hidden, "hidden"), (weight, "weight"), (teacher_logits, "teacher_logits"),
                  (loss_mask, "loss_mask")):
        _contig(t, nm)
    n, d = hidden.shape
    V = weight.shape[0]
    dt = _dtype_code(hidden)
    dev = hidden.device
    dirn = DIRECTIONS[direction] if isinstance(direction, str) else int(direction)
    scalars_out = scalars_out if scalars_out is not None else torch.empty(3, dtype=torch.float64, device=dev)
    per_token_out = per_token_out if per_token_out is not None else torch.empty(n, dtype=torch.float32, device=dev)
    lse_out = lse_out if lse_out is not None else torch.empty(n, dtype=torch.float32, device=dev)
    alloc = torch.zeros if flags & ACCUMULATE_GRADS else torch.empty
    if want_d_hidden and d_hidden is None:
        d_hidden = alloc(n, d, dtype=torch.float32, device=dev)
    if want_d_weight and d_weight is None:
        d_weight = alloc(V, d, dtype=torch.float32, device=dev)
    ws = _ws(ws, KIND_DISTILL, n, d, V, dt, dev)
    head = (n, d, V, n if chunk is None else chunk, dt, _ptr(hidden), _len(hidden), _ptr(weight),
            _len(weight), _ptr(teacher_logits), _len(teacher_logits), _ptr(loss_mask), dirn,
            temperature, z_weight, grad_scale)
    tail = (_ptr(scalars_out), _ptr(per_token_out), _ptr(lse_out), _ptr(d_hidden), _ptr(d_weight),
            _ptr(ws), ws.numel(), _stream(stream))
    if flags == 0:
        _check(lib.lossk_distill_fwd_bwd(*head, *tail), "lossk_distill_fwd_bwd")
    else:
        _check(lib.lossk_distill_fwd_bwd_ex(*head, flags, *tail), "lossk_distill_fwd_bwd_ex")
    return {"scalars": scalars_out, "per_token": per_token_out, "lse": lse_out,
            "d_hidden": d_hidden, "d_weight": d_weight}


def lossk_ce_chunk_invariance(hidden, weight, targets, loss_mask=None, z_weight=0.0, ws=None,
                              stream=None) -> float:
    """Max |difference| between lossk_ce_fwd at chunk 1 and at chunk n_tok (or the largest
    chunk the logit budget allows) over the scalars and every token's lse and ce."""
    for t, nm in ((hidden, "hidden"), (weight, "weight"), (targets, "targets"), (loss_mask, "loss_mask")):
        _contig(t, nm)
    n, d = hidden.shape
    V = weight.shape[0]
    dt = _dtype_code(hidden)
    ws = _ws(ws, KIND_CE_CHUNK_CHECK, n, d, V, dt, hidden.device)
    out = _dbl(-1.0)
    st = lib.lossk_ce_chunk_invariance(n, d, V, dt, _ptr(hidden), _len(hidden), _ptr(weight),
                                       _len(weight), _ptr(targets), _len(targets), _ptr(loss_mask),
                                       z_weight, ctypes.byref(out), _ptr(ws), ws.numel(),
                                       _stream(stream))
    _check(st, "lossk_ce_chunk_invariance")
    return out.value


def lossk_distill_from_logits(logits, teacher_logits, direction="fkl", temperature=1.0,
                              loss_mask=None, z_weight=0.0, grad_scale=1.0, flags=0, want_grad=True,
                              scalars_out=None, per_token_out=None, lse_out=None, grad_logits=None,
                              ws=None, stream=None):
    for t, nm in ((logits, "logits"), (teacher_logits, "teacher_logits"), (loss_mask, "loss_mask")):
        _contig(t, nm)
    n, V = logits.shape
    dt = _dtype_code(logits)
    dev = logits.device
    dirn = DIRECTIONS[direction] if isinstance(direction, str) else int(direction)
    scalars_out = scalars_out if scalars_out is not None else torch.empty(3, dtype=torch.float64, device=dev)
    per_token_out = per_token_out if per_token_out is not None else torch.empty(n, dtype=torch.float32, device=dev)
    lse_out = lse_out if lse_out is not None else torch.empty(n, dtype=torch.float32, device=dev)
    if want_grad and grad_logits is None:
        grad_logits = torch.zeros_like(logits) if flags & ACCUMULATE_GRADS else torch.empty_like(logits)
    ws = _ws(ws, KIND_FROM_LOGITS, n, 1, V, dt, dev)
    st = lib.lossk_distill_from_logits(n, V, dt, _ptr(logits), _len(logits), _ptr(teacher_logits),
                                       _len(teacher_logits), _ptr(loss_mask), dirn, temperature,
                                       z_weight, grad_scale, flags, _ptr(scalars_out),
                                       _ptr(per_token_out), _ptr(lse_out), _ptr(grad_logits),
                                       _len(grad_logits), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "lossk_distill_from_logits")
    return {"scalars": scalars_out, "per_token": per_token_out, "lse": lse_out,
            "grad_logits": grad_logits}


def lossk_device_status(ws, stream=None) -> int:
    return lib.lossk_device_status(_ptr(ws), ws.numel(), _stream(stream))


# ---- vocabulary-parallel cross-entropy ---------------------------------------------

def lossk_ce_shard_fwd(hidden, weight_shard, targets, v0, vocab_total, partials=None, ws=None, stream=None):
    """Partials float[3][n] of the shard holding vocabulary rows [v0, v0 + rows)."""
    for t, nm in ((hidden, "hidden"), (weight_shard, "weight_shard"), (targets, "targets")):
        _contig(t, nm)
    n, d = hidden.shape
    Vs = weight_shard.shape[0]
    dt = _dtype_code(hidden)
    dev = hidden.device
    partials = partials if partials is not None else torch.empty(3, n, dtype=torch.float32, device=dev)
    ws = _ws(ws, KIND_SHARD_FWD, n, d, Vs, dt, dev)
    st = lib.lossk_ce_shard_fwd(n, d, Vs, v0, vocab_total, dt, _ptr(hidden), _len(hidden), _ptr(weight_shard),
                                _len(weight_shard), _ptr(targets), _len(targets), _ptr(partials), _len(partials),
                                _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "lossk_ce_shard_fwd")
    return partials


def lossk_ce_shard_combine(partials_all, loss_mask=None, z_weight=0.0, lse_out=None, ce_out=None,
                           scalars_out=None, ws=None, stream=None):
    """lse, ce and the scalars from every shard's partials [P][3][n], in shard order."""
    _contig(partials_all, "partials_all")
    _contig(loss_mask, "loss_mask")
    P, three, n = partials_all.shape
    assert three == 3
    dev = partials_all.device
    lse_out = lse_out if lse_out is not None else torch.empty(n, dtype=torch.float32, device=dev)
    ce_out = ce_out if ce_out is not None else torch.empty(n, dtype=torch.float32, device=dev)
    scalars_out = scalars_out if scalars_out is not None else torch.empty(3, dtype=torch.float64, device=dev)
    ws = _ws(ws, KIND_SHARD_COMBINE, n, 1, 1, F32, dev)
    st = lib.lossk_ce_shard_combine(n, P, _ptr(partials_all), _len(partials_all), _ptr(loss_mask), z_weight,
                                    _ptr(lse_out), _ptr(ce_out), _ptr(scalars_out), _ptr(ws), ws.numel(),
                                    _stream(stream))
    _check(st, "lossk_ce_shard_combine")
    return {"lse": lse_out, "ce": ce_out, "scalars": scalars_out}


def lossk_ce_shard_bwd(hidden, weight_shard, targets, v0, vocab_total, lse, loss_mask=None, z_weight=0.0,
                       grad_scale=1.0, d_hidden=None, d_weight=None, want_d_hidden=True, want_d_weight=True,
                       ws=None, stream=None):
    """The shard's share of d_hidden and its d_weight rows, given the whole row's lse."""
    for t, nm in ((hidden, "hidden"), (weight_shard, "weight_shard"), (targets, "targets"), (lse, "lse"),
                  (loss_mask, "loss_mask")):
        _contig(t, nm)
    n, d = hidden.shape
    Vs = weight_shard.shape[0]
    dt = _dtype_code(hidden)
    dev = hidden.device
    if want_d_hidden and d_hidden is None:
        d_hidden = torch.empty(n, d, dtype=torch.float32, device=dev)
    if want_d_weight and d_weight is None:
        d_weight = torch.empty(Vs, d, dtype=torch.float32, device=dev)
    ws = _ws(ws, KIND_SHARD_BWD, n, d, Vs, dt, dev)
    st = lib.lossk_ce_shard_bwd(n, d, Vs, v0, vocab_total, dt, _ptr(hidden), _len(hidden), _ptr(weight_shard),
                                _len(weight_shard), _ptr(targets), _len(targets), _ptr(loss_mask), z_weight,
                                grad_scale, _ptr(lse), _len(lse), _ptr(d_hidden), _ptr(d_weight), _ptr(ws),
                                ws.numel(), _stream(stream))
    _check(st, "lossk_ce_shard_bwd")
    return {"d_hidden": d_hidden, "d_weight": d_weight}


def lossk_selftest_wait(n_stages: int, n_arrive: int, limit_ns: int, ws, stream=None):
    """Run the bounded-wait self-test; returns (status, stages the consumer saw)."""
    seen = _i32(0)
    st = lib.lossk_selftest_wait(n_stages, n_arrive, limit_ns, ctypes.byref(seen), _ptr(ws), ws.numel(),
                                 _stream(stream))
    return st, seen.value


# ---- tracing ------------------------------------------------------------------

def lossk_kernel_name(kind: int) -> str:
    return lib.lossk_kernel_name(kind).decode()


def lossk_launch_count() -> int:
    return lib.lossk_launch_count()


def lossk_profile_enable(on: bool = True) -> None:
    lib.lossk_profile_enable(1 if on else 0)


def lossk_profile_read(reset: bool = True) -> dict:
    """{kernel name: (total ms, launches)} for the kernels launched while profiling."""
    ms = (_dbl * N_KERNELS)()
    cnt = (_i64 * N_KERNELS)()
    k = lib.lossk_profile_read(ms, cnt, N_KERNELS, 1 if reset else 0)
    if k < 0:
        raise LosskError(589, "lossk_profile_read")
    return {lossk_kernel_name(i): (ms[i], cnt[i]) for i in range(k) if cnt[i]}
