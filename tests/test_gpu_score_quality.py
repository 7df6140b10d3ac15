"""Score quality of mse-only keys versus prod keys at equal bits (needs a GPU).

The page's community finding #1: QJL removes the inner-product bias but adds
variance, and softmax amplifies variance, so mse-only keys often match the top
token better.  bench.py --study score-quality reports the full table; this test
checks what the theory fixes about the scores the decode kernel produces:
  mse   slope of the quantized scores on the exact ones is 1 − D_mse(b), and the
        remaining relative noise power is D_mse(b)·(1 − D_mse(b));
  prod  slope 1 (unbiased), noise power at most (π/2)·D_mse(b − 1) (Theorem 2),
        and more noise than mse at the same b.
"""
import math

import pytest

import bench
import oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tq():
    import kv_cache_vector_18_b300 as m
    return m


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_score_slope_and_noise(tq, bits):
    d = 128
    m = bench.score_quality(tq, d, bits, "mse", 4.0, B=2, seed=7 + bits)
    p = bench.score_quality(tq, d, bits, "prod", 4.0, B=2, seed=7 + bits)
    dm = O.mse_distortion_theory(d, 1 << bits)
    dp = O.mse_distortion_theory(d, 1 << (bits - 1))
    assert abs(m["score_slope"] - (1 - dm)) <= 0.02, (m, dm)
    assert abs(m["score_noise"] ** 2 / (dm * (1 - dm)) - 1) <= 0.15, (m, dm)
    assert abs(p["score_slope"] - 1) <= 0.03, p
    assert p["score_noise"] ** 2 <= 1.1 * (math.pi / 2) * dp, (p, dp)
    assert p["score_noise"] > m["score_noise"]
    for r in (m, p):
        assert 0.0 <= r["top1"] <= 1.0 and 0.0 <= r["top5_recall"] <= 1.0
        assert r["kl"] >= 0.0 and math.isfinite(r["out_rel_l2"])
