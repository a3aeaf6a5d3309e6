"""Writes the oracle's values for the two largest workloads at their full size.

    python tests/golden/make_full_size_goldens.py [ce_z | distill | all]

At n_tok 8192, d_model 4096, vocab 128256 (cross-entropy + z-loss, 5 % of the
tokens masked) and at n_tok 4096, d_model 2048, vocab 151936 (distillation
against a bf16 teacher at T = 2, 10 % masked, z-loss), the fp64 oracle needs
minutes on a CPU, too long for a GPU test.  This script runs it once and
stores what the full-size parity tests compare against:

  every token's lse and loss, the three reduced scalars, and the d_weight rows
  of a fixed sample of vocabulary rows (every sampled row over every token).

Only ``oracle/`` computes these values; ``lossk_inputs`` draws the inputs
(the same seeded recipe the tests use), and a SHA-256 fingerprint of those
inputs is stored beside the values so that a test run on another machine can
tell whether it drew the same inputs.  d_weight rows are stored as float32
(the tolerance they are held to is 1e-2 relative L2); everything else as
float64.
"""
from __future__ import annotations

import hashlib
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import lossk_inputs as li  # noqa: E402
import oracle  # noqa: E402

CE_Z = "ce_z_8192x4096x128256"
DISTILL = "distill_z_4096x2048"
N_VROWS = 16


def golden_path(name: str) -> str:
    return os.path.join(HERE, f"full_size_{name}.npz")


def fingerprint(x: dict) -> str:
    """SHA-256 over the inputs' bytes, in a fixed key order."""
    h = hashlib.sha256()
    for k in ("hidden", "weight", "targets", "mask", "teacher"):
        a = x.get(k)
        if a is None:
            continue
        h.update(k.encode())
        h.update(np.ascontiguousarray(a).tobytes())
    return h.hexdigest()


def sample_vrows(V: int, targets=None) -> np.ndarray:
    """The first and last vocabulary rows, some target rows, the rest random."""
    g = np.random.default_rng(2024)
    picks = [0, V - 1]
    if targets is not None:
        picks += [int(v) for v in np.unique(targets)[:: max(1, len(np.unique(targets)) // 6)][:6]]
    while len(picks) < N_VROWS:
        v = int(g.integers(0, V))
        if v not in picks:
            picks.append(v)
    return np.array(sorted(picks[:N_VROWS]), dtype=np.int64)


def make_ce_z() -> None:
    w = li.WORKLOADS[CE_Z]
    x = li.make(w)
    t0 = time.time()
    f = oracle.ce_fwd(x["hidden"], x["weight"], x["targets"], mask=x["mask"], chunk=w.chunk,
                      z_weight=w.z_weight)
    t1 = time.time()
    vrows = sample_vrows(w.vocab, x["targets"])
    dw = oracle.ce_dweight_rows(x["hidden"], x["weight"], x["targets"], f["lse"], vrows,
                                mask=x["mask"], z_weight=w.z_weight)
    np.savez_compressed(golden_path(CE_Z), fingerprint=np.array(fingerprint(x)), lse=f["lse"],
                        ce=f["ce"], scalars=np.array([f["total"], f["ce_mean"], f["z_mean"]]),
                        vrows=vrows, dweight_rows=dw.astype(np.float32))
    print(f"{CE_Z}: forward {t1 - t0:.0f} s, d_weight rows {time.time() - t1:.0f} s")


def make_distill() -> None:
    w = li.WORKLOADS[DISTILL]
    x = li.make(w)
    vrows = sample_vrows(w.vocab)
    out = {"fingerprint": np.array(fingerprint(x)), "vrows": vrows}
    allrows = np.arange(w.n_tok)
    for direction in ("ce", "fkl", "rkl"):
        t0 = time.time()
        r = oracle.distill_token_rows(x["hidden"], x["weight"], x["teacher"], direction, allrows,
                                      temperature=w.temperature, mask=x["mask"],
                                      z_weight=w.z_weight, want_dh=False)
        s = oracle.reduce_tokens(r["loss"], r["lse"], mask=x["mask"], z_weight=w.z_weight)
        dw = oracle.distill_dweight_rows(x["hidden"], x["weight"], x["teacher"], direction, r["lse"],
                                         r["loss"], vrows, temperature=w.temperature, mask=x["mask"],
                                         z_weight=w.z_weight)
        out[f"{direction}_lse"] = r["lse"]
        out[f"{direction}_loss"] = r["loss"]
        out[f"{direction}_scalars"] = np.array([s["total"], s["loss_mean"], s["z_mean"]])
        out[f"{direction}_dweight_rows"] = dw.astype(np.float32)
        print(f"{DISTILL} {direction}: {time.time() - t0:.0f} s")
    np.savez_compressed(golden_path(DISTILL), **out)


if __name__ == "__main__":
    which = sys.argv[1] if len(sys.argv) > 1 else "all"
    if which in ("ce_z", "all"):
        make_ce_z()
    if which in ("distill", "all"):
        make_distill()
