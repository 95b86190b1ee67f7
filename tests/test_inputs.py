"""The seeded input module: layouts that several callers derive from one
workload must agree with the oracle's own reading of the page table."""
import numpy as np
import torch

import workloads
from oracle import attention as oatt
from oracle.numerics import decode_e4m3


def test_contiguous_rope_rows_are_the_paged_rows():
    w = workloads.custom([5, 0, 3, 20], [2, 6, 4, 9], heads=1, page_size=4, seed=3,
                         row_width=80, rope_col=16)
    rows, scales = workloads.contiguous_rope(w)
    assert rows.shape == (w.total_k, 80) and scales is None
    G = 0
    for b in range(w.batch):
        L = int(w.n[b] + w.prior[b])
        got = rows[G:G + L, 16:80].float().numpy()
        assert np.array_equal(got, oatt.gather_k_rope(w, b)), b
        G += L


def test_contiguous_rope_fp8_scales_follow_rows():
    w = workloads.custom([7, 2], [3, 5], heads=1, page_size=4, seed=4, dtype="fp8")
    rows, scales = workloads.contiguous_rope(w)
    deq = decode_e4m3(rows.view(torch.uint8).numpy()) * scales.numpy()[:, None]
    G = 0
    for b in range(w.batch):
        L = int(w.n[b] + w.prior[b])
        assert np.array_equal(deq[G:G + L, :64], oatt.gather_k_rope(w, b)), b
        G += L
