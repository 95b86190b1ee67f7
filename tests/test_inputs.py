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


def test_per_token_k_requantises_each_row_to_its_own_amax():
    w = workloads.custom([9, 4], [3, 6], heads=2, page_size=4, seed=5, dtype="fp8")
    wt = workloads.per_token_k(w)
    ks = np.asarray(wt.k_scale)
    assert ks.shape == (w.total_k,) and ks.dtype == np.float32 and (ks > 0).all()
    codes = decode_e4m3(wt.k_nope.view(torch.uint8).numpy()).reshape(w.total_k, -1)
    # Every row uses its full range: its largest code is the e4m3 maximum.
    assert np.array_equal(np.abs(codes).max(axis=1), np.full(w.total_k, 448.0))
    # Row values follow the per-tensor ones times a per-row factor in [1/4, 4],
    # up to e4m3 rounding (relative 2^-4 plus the subnormal step of the row).
    old = decode_e4m3(w.k_nope.view(torch.uint8).numpy()).reshape(w.total_k, -1) * w.k_scale
    new = codes * ks[:, None]
    big = np.abs(old) > 0.25 * np.abs(old).max(axis=1, keepdims=True)
    ratio = np.where(big, new / np.where(big, old, 1.0), np.nan)
    f = np.nanmedian(ratio, axis=1)
    assert ((f >= 0.25 * 0.9) & (f <= 4.0 * 1.1)).all()
    assert np.nanmax(np.abs(ratio / f[:, None] - 1.0)) < 0.15
    # Everything but K_nope and its scale is the original workload's.
    assert wt.q is w.q and wt.v is w.v and wt.k_rope_pool is w.k_rope_pool
