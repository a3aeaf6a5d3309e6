"""Failure detection on the GPU without a fault: a bounded device wait that
runs out.

Every wait in the tensor-core kernels gives up after a time limit, records a
timeout in the workspace's error word and lets the kernel unwind.  Here a
producer deliberately skips two of its four barrier arrivals, so the
consumer's wait runs out after 5 ms (no trap, no endless loop, no bad
address): the call reports 590, the error word stays set until
lossk_device_status reads and clears it, and the next call on the same
workspace runs clean.
"""
import time

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    from conftest import build_lib
    build_lib()
    import output_projection_cross_gb300 as L
    assert torch.cuda.is_available()
    return L


def test_every_stage_arrives(L):
    ws = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    assert L.lossk_selftest_wait(4, 4, 5_000_000, ws) == (580, 4)
    assert L.lossk_device_status(ws) == 580


def test_a_wait_that_runs_out_reports_590_and_the_next_call_runs_clean(L):
    ws = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    y = torch.zeros(64, dtype=torch.int64, device="cuda")
    t0 = time.perf_counter()
    st, seen = L.lossk_selftest_wait(4, 2, 5_000_000, ws)
    dt = time.perf_counter() - t0
    assert (st, seen) == (590, 2)
    assert dt >= 0.005                      # the consumer waited out its limit ...
    assert dt < 5.0                         # ... and no longer: the block unwound
    # until it is read, the error word makes every call on this workspace report it
    assert L.lib.lossk_targets_check(64, 10, y.data_ptr(), 64, ws.data_ptr(), ws.numel(),
                                     torch.cuda.current_stream().cuda_stream) == 590
    assert L.lossk_device_status(ws) == 590
    assert L.lossk_device_status(ws) == 580                 # read and cleared
    assert L.lib.lossk_targets_check(64, 10, y.data_ptr(), 64, ws.data_ptr(), ws.numel(),
                                     torch.cuda.current_stream().cuda_stream) == 580
    # the context is unharmed: a full call still matches its own rerun
    X = torch.randn(8, 100, device="cuda").to(torch.bfloat16)
    yy = torch.randint(0, 100, (8,), device="cuda")
    a = L.lossk_ce_from_logits(X, yy, want_grad=True)
    b = L.lossk_ce_from_logits(X, yy, want_grad=True)
    torch.cuda.synchronize()
    assert torch.equal(a["lse"], b["lse"]) and torch.equal(a["grad_logits"], b["grad_logits"])


def test_selftest_refuses_bad_arguments(L):
    ws = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    assert L.lossk_selftest_wait(0, 0, 5_000_000, ws)[0] == 582
    assert L.lossk_selftest_wait(9, 0, 5_000_000, ws)[0] == 582
    assert L.lossk_selftest_wait(4, 5, 5_000_000, ws)[0] == 582
    assert L.lossk_selftest_wait(4, 2, 10, ws)[0] == 585
    assert L.lossk_selftest_wait(4, 2, 2_000_000_000, ws)[0] == 585
    assert L.lossk_device_status(ws) == 580                 # nothing ran
