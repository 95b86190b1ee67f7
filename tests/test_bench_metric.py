"""The throughput metric bench.py reports: causal-effective flops count every
visible (query, key, head) triple once at 2 * (192 + 128) flops (QK^T and PV
multiply-adds), checked here against a brute-force count of visible pairs."""
import numpy as np
import pytest

import bench
import workloads


def _visible_pairs(w):
    total = 0
    for b in range(w.batch):
        n, prior = int(w.n[b]), int(w.prior[b])
        L = n + prior
        i = np.arange(n)[:, None]
        j = np.arange(L)[None, :]
        allowed = (j <= prior + i) if w.spec.mask == "causal" else np.ones((n, L), dtype=bool)
        total += int(allowed.sum())
    return total


@pytest.mark.parametrize("mask", ["causal", "null"])
@pytest.mark.parametrize("seed", [1, 2, 3])
def test_causal_flops_counts_visible_pairs(mask, seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 6))
    n = rng.integers(0, 300, size=B).tolist()
    prior = rng.integers(0, 400, size=B).tolist()
    w = workloads.custom(n, prior, heads=3, seed=seed, mask=mask)
    assert bench.causal_flops(w) == 3 * 2 * 320 * _visible_pairs(w)


def test_oracle_sample_flops_match_its_rows():
    w = workloads.custom([40, 90, 10], [5, 20, 0], heads=2, seed=4)
    f, dt, text = bench.oracle_sample(w, 25, [0, 1])
    b = int(np.argmax(w.n))
    n, prior = int(w.n[b]), int(w.prior[b])
    pairs = sum(prior + i + 1 for i in range(n - 25, n))     # the last 25 rows of sequence b
    assert f == 2 * 320 * pairs * 2 and dt > 0 and "last 25 query rows" in text


def test_peaks_file_or_fallback():
    peaks, src = bench.load_peaks()
    assert src in ("measured", "fallback")
    assert peaks["bf16_tflops"] > 100 and peaks["hbm_gbs"] > 1000
