"""Pins for the chunked-execution oracle (one attention call per buffer row of
generic_flare_mla_prefill_ragged_paged_plan, rows combined by log-sum-exp).

* Mathematics: splitting the keys of a softmax into disjoint sets and
  combining the per-set results by their log-sum-exp reproduces the softmax
  over all keys.  So the merge of the plan's rows must equal the full-context
  oracle (itself pinned to torch's scaled_dot_product_attention) for every
  buffer size, including one key per row; a wrong lse (missing scale, log2 in
  place of ln, a dropped max) or a wrong absolute position (mask or page
  lookup off by the row's cache offset) breaks that equality.
* Closed form: with Q = 0 every visible score is 0, so lse = ln(number of
  visible keys) and the output is the mean of the visible V rows; counted and
  summed here one key at a time in Python.
* Degenerate cases: a row that covers the whole context is the full-context
  call; a query with no visible key in a row gets 0 and -inf.
"""
import math

import numpy as np
import pytest

import workloads
from oracle import attention as oatt
from oracle import chunked as och
from oracle import plan as oplan
from oracle.numerics import decode_bf16


def _rows(w, T):
    R_max = oplan.num_rows(w.row_offsets, w.prior, T)
    bro, co, blen, R = oplan.plan_formula(w.row_offsets, w.prior, T, R_max)
    return [(bro[r], co[r]) for r in range(R)]


def _merged(w, T, heads=None):
    parts = [och.window_reference(w, bro, co, heads) for bro, co in _rows(w, T)]
    return och.merge([o for o, _ in parts], [l for _, l in parts])


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("mask", ["causal", "null"])
@pytest.mark.parametrize("T", [1, 3, 7, 16, 40, 1000])
def test_merge_of_plan_rows_equals_full_context(dtype, mask, T):
    w = workloads.custom([5, 1, 0, 9, 12], [0, 3, 2, 6, 17], heads=2, page_size=4, dtype=dtype,
                         seed=11, mask=mask)
    ref = oatt.reference(w)
    got = _merged(w, T)
    assert np.isfinite(got).all()
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12)


def test_merge_tiny_config_rows():
    w = workloads.generate(workloads.config("tiny_bf16"))
    np.testing.assert_allclose(_merged(w, w.spec.buffer_token_size), oatt.reference(w),
                               rtol=1e-11, atol=1e-12)


def test_single_row_is_full_context_call():
    w = workloads.custom([6, 4], [3, 0], heads=2, page_size=4, seed=12)
    rows = _rows(w, 10_000)
    assert len(rows) == 1
    out, lse = och.window_reference(w, *rows[0])
    np.testing.assert_allclose(out, oatt.reference(w), rtol=1e-12, atol=1e-12)
    assert np.isfinite(lse).all()


@pytest.mark.parametrize("mask", ["causal", "null"])
def test_zero_queries_give_counts_and_means(mask):
    w = workloads.custom([7, 3, 5], [4, 0, 9], heads=2, page_size=4, seed=13, mask=mask)
    w.q.zero_()
    v = decode_bf16(w.v.view(__import__("torch").int16).numpy().view(np.uint16))
    L = w.n + w.prior
    G = np.concatenate([[0], np.cumsum(L)])
    for bro, co in _rows(w, 6):
        out, lse = och.window_reference(w, bro, co)
        for b in range(w.batch):
            W = int(bro[b + 1]) - int(bro[b])
            for i in range(int(w.n[b])):
                t = int(w.row_offsets[b]) + i
                if W == 0:
                    assert np.isnan(lse[t]).all()
                    continue
                vis = [a for a in range(int(co[b]), int(co[b]) + W)
                       if mask == "null" or a <= int(w.prior[b]) + i]
                for h in range(w.heads):
                    if not vis:
                        assert lse[t, h] == -math.inf
                        assert (out[t, h] == 0).all()
                        continue
                    assert lse[t, h] == pytest.approx(math.log(len(vis)), abs=1e-12)
                    mean = [sum(v[G[b] + a, h, d] for a in vis) / len(vis) for d in range(128)]
                    np.testing.assert_allclose(out[t, h], mean, rtol=1e-12, atol=1e-12)


def test_query_without_visible_key():
    # prior 0, 6 new tokens; a row holding positions 4..5 only: queries 0..3 see nothing.
    w = workloads.custom([6], [0], heads=1, page_size=4, seed=14)
    out, lse = och.window_reference(w, [0, 2], [4])
    assert (lse[:4, 0] == -math.inf).all() and (out[:4] == 0).all()
    assert np.isfinite(lse[4:]).all()


def test_merge_skips_absent_and_empty_rows():
    rng = np.random.default_rng(0)
    o = rng.normal(size=(3, 2, 128))
    l = rng.normal(size=(3, 2))
    nan_o = np.full_like(o, np.nan)
    nan_l = np.full_like(l, np.nan)
    ninf_l = np.full_like(l, -np.inf)
    np.testing.assert_allclose(och.merge([o, nan_o], [l, nan_l]), o, rtol=1e-15)
    np.testing.assert_allclose(och.merge([o, np.zeros_like(o)], [l, ninf_l]), o, rtol=1e-15)
    # Equal weights average; a weight e^1 : e^0 mixes e/(1+e) : 1/(1+e).
    o2 = rng.normal(size=o.shape)
    np.testing.assert_allclose(och.merge([o, o2], [l, l]), (o + o2) / 2, rtol=1e-13)
    e = math.e
    np.testing.assert_allclose(och.merge([o, o2], [l + 1, l]), (e * o + o2) / (1 + e), rtol=1e-13)
    assert np.isnan(och.merge([nan_o], [nan_l])).all()
