"""The seeded input generator: deterministic, and drawing what its recipe says."""
import numpy as np

import lossk_inputs as li


def test_deterministic_and_independent_streams():
    a = li.make("tiny_fp32_ce", seed=0)
    b = li.make("tiny_fp32_ce", seed=0)
    for k in ("hidden", "weight", "targets"):
        assert np.array_equal(a[k], b[k])
    c = li.make("tiny_fp32_ce", seed=0, vocab=500)       # other shape, same hidden
    assert np.array_equal(a["hidden"], c["hidden"])
    assert a["weight"].dtype == np.float32 and a["targets"].dtype == np.int64


def test_bf16_rounding_is_exact_bf16():
    h = li.hidden(0, 8, 16, dtype="bf16")
    bits = h.view(np.uint32)
    assert np.all(bits & 0xFFFF == 0)                      # low mantissa half is zero


def test_distributions():
    w = li.weight(0, 4000, 64, std=0.02, dtype="fp32")
    assert abs(w.std() - 0.02) < 0.0005 and abs(w.mean()) < 0.0005
    y = li.targets(0, 200000, 151936, "zipf1.1")
    assert y.min() >= 0 and y.max() < 151936
    p = np.arange(1, 151937, dtype=np.float64) ** -1.1
    p /= p.sum()
    assert abs((y == 0).mean() - p[0]) < 0.01 and abs((y == 1).mean() - p[1]) < 0.01
    u = li.targets(0, 100000, 1000, "uniform")
    assert abs(u.mean() - 499.5) < 5
    m = li.mask(0, 8192, 0.05)
    assert (m == 0).sum() == 410 and m.dtype == np.uint8
    assert (li.mask(0, 4096, 0.10) == 0).sum() == 410
